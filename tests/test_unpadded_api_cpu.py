"""The unpadded-tensor layer of the binding (attn_self, attn_cross, attn_sharded, rope)
without a GPU: its padding plan and every argument check that comes before a device call."""
import os

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def api():
    if not os.path.exists(os.path.join(ROOT, "video_dit_attention_gb300", "libdit_attn.so")):
        from video_dit_attention_gb300.build import build
        build()
    from video_dit_attention_gb300 import dit_attn
    return dit_attn


def _t(*shape):
    return torch.zeros(shape, dtype=torch.bfloat16)


@pytest.mark.parametrize("n,padded", [(0, 128), (1, 128), (128, 128), (129, 256), (300, 384), (4680, 4736),
                                      (9384, 9472), (75600, 75648)])
def test_padding_is_whole_tiles_and_at_least_one(api, n, padded):
    assert api._tiles(n) == padded


def test_attn_self_rejects_bad_options_before_any_device_call(api):
    q, k = _t(1, 300, 2, 128), _t(1, 333, 2, 128)
    with pytest.raises(ValueError, match="mode"):
        api.attn_self(q, k, k, "1d", mode="bf16")
    with pytest.raises(ValueError, match="T\\*Hh\\*W"):
        api.attn_self(q, k, k, (3, 10, 10))
    with pytest.raises(ValueError, match="T\\*Hh\\*W"):
        api.attn_self(q, q, q, (3, 10, 11))
    with pytest.raises(ValueError, match="RMSNorm"):
        api.attn_self(q, k, k, None, norm_q=torch.ones(128), norm_k=torch.ones(128))
    with pytest.raises(ValueError, match="RMSNorm"):
        api.attn_self(q, k, k, "1d", mode="fp8", norm_q=torch.ones(128), norm_k=torch.ones(128))
    with pytest.raises(ValueError, match="both"):
        api.attn_self(q, k, k, "1d", norm_q=torch.ones(128))
    with pytest.raises(ValueError, match="fixed-m"):
        api.attn_self(q, k, k, None, mode="fixed_m")
    with pytest.raises(ValueError, match="matching"):
        api.attn_self(q, _t(1, 333, 3, 128), _t(1, 333, 3, 128))
    with pytest.raises(ValueError, match="CUDA"):
        api.attn_self(q, k, k, "1d")          # valid options, host tensors: no CPU path


def test_attn_cross_checks_lengths(api):
    q, k = _t(2, 300, 2, 128), _t(2, 512, 2, 128)
    with pytest.raises(ValueError, match="kv_valid_len"):
        api.attn_cross(q, k, k, [10])
    with pytest.raises(ValueError, match="kv_valid_len"):
        api.attn_cross(q, k, k, [10, 513])
    with pytest.raises(ValueError, match="kv_valid_len"):
        api.attn_cross(q, k, k, [-1, 3])
    with pytest.raises(ValueError, match="512"):
        api.attn_cross(q, _t(2, 513, 2, 128), _t(2, 513, 2, 128), [1, 1])
    with pytest.raises(ValueError, match="CUDA"):
        api.attn_cross(q, k, k, [512, 0])


def test_attn_sharded_and_rope_check_their_options(api):
    q, k = _t(1, 100, 2, 64), _t(1, 200, 2, 64)
    with pytest.raises(ValueError, match="rope"):
        api.attn_sharded(q, [(k, k)], rope=(1, 10, 20))
    with pytest.raises(ValueError, match="shards"):
        api.attn_sharded(q, [])
    with pytest.raises(ValueError, match="shard 1"):
        api.attn_sharded(q, [(k, k), (k, _t(1, 199, 2, 64))])
    with pytest.raises(ValueError, match="CUDA"):
        api.attn_sharded(q, [(k, k)])
    with pytest.raises(ValueError, match="rope"):
        api.rope(q, None)
    with pytest.raises(ValueError, match="T\\*Hh\\*W"):
        api.rope(q, (2, 5, 11))
    with pytest.raises(ValueError, match="CUDA"):
        api.rope(q, "1d")
