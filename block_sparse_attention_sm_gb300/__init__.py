"""Skip-softmax (BLASST) attention for GB300 (sm_103a)."""
