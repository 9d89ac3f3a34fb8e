"""GB300-native context-parallel causal attention (tile attention + LSE merge).

The compute lives in ``libcpattn.so`` (hand-written CUDA for sm_103a behind a
C ABI, declared in ``include/cpattn.h``).  This package only marshals
arguments: see ``tile_attention_lse_gb300.api``.
"""
