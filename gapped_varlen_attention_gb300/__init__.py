"""Gapped variable-length attention forward for GB300 (sm_103a)."""
