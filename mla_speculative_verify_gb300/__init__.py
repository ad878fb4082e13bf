"""GB300 (sm_103a) MLA speculative-verify decode behind a C-ABI library."""
