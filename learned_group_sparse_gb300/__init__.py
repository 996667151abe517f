"""Focus attention inference path for GB300 (sm_103a)."""
