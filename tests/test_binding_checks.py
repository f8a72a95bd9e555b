"""The torch helpers refuse tensors the kernels would misread, before any launch.

The library takes raw device addresses with a fixed layout; the helpers in
block_sparse_attention_sm_gb300 check element type, contiguity, shape, size
and device first.  Everything here raises on the host, so it runs without a
GPU (the device check comes last, after the others have passed).
"""
import pytest
import torch

import block_sparse_attention_sm_gb300 as ss

BF = torch.bfloat16


def _qkv(B=1, Hq=2, Hkv=1, L=256, d=64, dtype=BF):
    q = torch.zeros(B, Hq, L, d, dtype=dtype)
    k = torch.zeros(B, Hkv, L, d, dtype=dtype)
    return q, k, k.clone()


def test_prefill_rejects_host_tensors():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="CUDA tensor"):
        ss.prefill(q, k, v, scale=0.125)


def test_prefill_rejects_other_element_types():
    q, k, v = _qkv(dtype=torch.float16)
    with pytest.raises(ValueError, match="element type"):
        ss.prefill(q, k, v, scale=0.125)


def test_prefill_rejects_strided_views():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="contiguous"):
        ss.prefill(q.transpose(2, 3), k, v, scale=0.125)


def test_prefill_rejects_mismatched_shapes_and_short_buffers():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="shape of k"):
        ss.prefill(q, k, v[:, :, :128].contiguous(), scale=0.125)
    with pytest.raises(ValueError, match="at least 4 elements"):  # 1 * 2 heads * 2 blocks
        ss.prefill(q, k, v, scale=0.125, counts=torch.zeros(3, dtype=torch.int32))
    with pytest.raises(ValueError, match="element type"):
        ss.prefill(q, k, v, scale=0.125, counts=torch.zeros(4, dtype=torch.int64))
    with pytest.raises(ValueError, match="at least 8 elements"):  # 4 units x 2 tiles
        ss.prefill(q, k, v, scale=0.125, skip_mask=torch.zeros(7, dtype=torch.uint8))
    with pytest.raises(ValueError, match="expected shape"):
        ss.prefill(q, k, v, scale=0.125, out=torch.zeros(1, 2, 128, 64, dtype=BF))


def test_decode_checks():
    q = torch.zeros(2, 8, 128, dtype=BF)
    k = torch.zeros(2, 2, 300, 128, dtype=BF)
    with pytest.raises(ValueError, match="3 dimensions"):
        ss.decode(q[None], k, k, scale=0.1)
    with pytest.raises(ValueError, match="decode expects"):
        ss.decode(q[:1].contiguous(), k, k, scale=0.1)
    with pytest.raises(ValueError, match="at least 12 elements"):  # 2 seq x 2 heads x 3 splits
        ss.decode(q, k, k, scale=0.1, num_kv_splits=3, counts=torch.zeros(11, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        ss.decode(q, k, k, scale=0.1)


def test_mla_decode_checks():
    q = torch.zeros(2, 16, 576, dtype=BF)
    kv = torch.zeros(2, 300, 576, dtype=BF)
    with pytest.raises(ValueError, match="expected shape"):
        ss.mla_decode(q, kv, scale=0.07, out=torch.zeros(2, 16, 576, dtype=BF))
    with pytest.raises(ValueError, match="element type"):
        ss.mla_decode(q, kv.float(), scale=0.07)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ss.mla_decode(q, kv, scale=0.07)


def test_calibrate_checks():
    q, k, v = _qkv()
    with pytest.raises(ValueError, match="unknown kind"):
        ss.calibrate("encode", q, k, v, scale=0.125, target_sparsity=0.5)
    with pytest.raises(ValueError, match="3 dimensions"):  # decode takes q [B,Hq,d]
        ss.calibrate("decode", q, k, v, scale=0.125, target_sparsity=0.5)
    with pytest.raises(ValueError, match="at least 4 elements"):
        ss.calibrate("prefill", q, k, v, scale=0.125, target_sparsity=0.5,
                     counts=torch.zeros(2, dtype=torch.int32))
    with pytest.raises(ValueError, match="CUDA tensor"):
        ss.calibrate("prefill", q, k, v, scale=0.125, target_sparsity=0.5)


def test_well_formed_decode_and_latent_calibration_reach_the_device_check():
    q = torch.zeros(2, 8, 128, dtype=BF)
    k = torch.zeros(2, 2, 300, 128, dtype=BF)
    with pytest.raises(ValueError, match="q: must be a CUDA tensor"):
        ss.calibrate("decode", q, k, k.clone(), scale=0.1, target_sparsity=0.5, num_kv_splits=2)
    ql = torch.zeros(2, 16, 576, dtype=BF)
    kv = torch.zeros(2, 300, 576, dtype=BF)
    with pytest.raises(ValueError, match="q: must be a CUDA tensor"):
        ss.calibrate("mla_decode", ql, kv, None, scale=0.07, target_sparsity=0.5)
