"""Packed-sequence flash attention for GB300 (sm_103a)."""
