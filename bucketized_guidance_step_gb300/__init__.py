"""Fused guided denoise step for GB300 (sm_103a): C-ABI library and its Python binding."""
