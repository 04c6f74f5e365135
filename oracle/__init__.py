"""CPU oracle for the ZeRO-1 step (test infrastructure; never imported by the library)."""
