"""Batch-invariant mHC pre "H Aggregate" for GB300 (sm_103a)."""
