"""GB300-native video-DiT attention: split-halves RoPE, tile-padded self-attention with
exact pad-key masking, short-KV cross-attention and the LSE merge of key-shard partials.

The compute runs in hand-written sm_103a CUDA kernels behind a C-ABI shared library
(``include/dit_attn.h``). ``dit_attn`` is the thin Python binding over that library (it
raises at import if the library is missing; there is no CPU fallback). ``padding`` holds
the host-side padding plan, ``inputs`` the seeded synthetic input generators.
"""

__all__ = ["dit_attn", "padding", "inputs"]
