"""LLM.int8() mixed-precision decomposed matmul on one B300 (sm_103a)."""
