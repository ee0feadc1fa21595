"""Paged KV-cache attention for GB300 (sm_103a)."""
