"""CPU oracle of the Polestar calibration + commit path (test infrastructure only)."""
