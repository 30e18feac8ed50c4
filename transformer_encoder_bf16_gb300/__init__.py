"""Laya BF16 encoder forward pass on one GB300 (sm_103a): Python binding."""
