"""Host-side token padding plan (no device work).

The pages pad a video token sequence so that every shard (or the whole sequence) is a
whole number of kernel tiles, mask the pad keys inside attention, and cut the pad rows at
the end: Difflet PR #153 pads Wan's 4680 rows to 4736 (each of the 2 x tp ring halves a
multiple of 16 rows) and LTX-2's 2310 to 2312 (a multiple of 2 x tp); maxdiffusion PR #491
pads 75,600 tokens to 75,776 (each of CP = 4 shards a multiple of 128). On one GPU the
sequence is one shard and the tile is 128 rows.
"""
from __future__ import annotations

TILE = 128


def plan_token_padding(seq_len: int, multiple: int = TILE, shards: int = 1) -> int:
    """Padded length: `shards` equal shards, each rounded up to a multiple of `multiple`."""
    if seq_len < 0 or multiple < 1 or shards < 1:
        raise ValueError(f"bad padding plan: seq_len={seq_len} multiple={multiple} shards={shards}")
    per_shard = -(-seq_len // shards)
    return shards * (-(-per_shard // multiple) * multiple)
