"""Exact tiled attention with online softmax for GB300 (sm_103a)."""
