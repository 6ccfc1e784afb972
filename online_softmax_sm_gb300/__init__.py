"""Single-pass online-softmax attention forward for GB300 (sm_103a)."""
