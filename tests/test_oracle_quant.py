"""Pins for the oracle's NVFP4 (Q, K) and MXFP4 (V along keys) quantizers.

Checked against hand-worked blocks (tests/golden), the no-clip power-of-two
rule amax <= 6*2^e < 2*amax, and the per-element error bound of
round-to-nearest on the E2M1 grid.
"""
import json
import os

import numpy as np
import torch

import oracle
from blackwell_nvfp4_quantize_gb300 import workloads as wl

E2M1 = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])


def _bits(values, shape):
    t = torch.tensor(values, dtype=torch.float32).reshape(shape).to(torch.bfloat16)
    assert torch.equal(t.float().reshape(-1), torch.tensor(values, dtype=torch.float32)), "not bf16-exact"
    return wl.bf16_bits(t)


def _nib(payload_row, i):
    b = payload_row[i // 2]
    return (b & 0xF) if i % 2 == 0 else (b >> 4)


def _dec_codes(codes):
    codes = np.asarray(codes)
    v = E2M1[codes & 7]
    return np.where(codes & 8, -v, v)


def test_nvfp4_hand_worked(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "nvfp4_block.json")))
    B, H, N, D = gold["shape"]
    x = _bits(gold["values"], (B, H, N, D))
    payload, sf, g = oracle.quant_nvfp4(x, threads=1)
    assert g == np.float32(gold["g"])
    codes = [_nib(payload[0, 0, 0], i) for i in range(D)]
    assert codes == gold["codes"]
    for kb, want in enumerate(gold["sf_by_block"]):
        assert sf[oracle.sf_index(0, 1, 0, kb, D // 16)] == want, kb


def test_sf_atom_layout_is_a_bijection():
    # every (row, block) of one 128-row tile with 8 blocks maps to a distinct byte
    seen = set()
    for r in range(128):
        for kb in range(8):
            seen.add(oracle.sf_index(0, 1, r, kb, 8))
    assert seen == set(range(1024))
    assert oracle.sf_index(0, 1, 33, 5, 8) == 512 + 1 * 16 + 1 * 4 + 1
    assert oracle.sf_index(3, 2, 130, 0, 4) == (3 * 2 + 1) * 512 + 2 * 16


def test_nvfp4_error_bound_and_scales():
    q, _, _ = wl.make_custom(2, 3, 200, 64, seed=5, kind="wide")
    x = wl.bf16_bits(q)
    payload, sf, g = oracle.quant_nvfp4(x)
    xf = q.float().numpy()
    B, H, N, D = x.shape
    amax = np.abs(xf).max()
    assert g == np.float32(amax / np.float32(2688.0))
    for bh in range(B * H):
        b, h = divmod(bh, H)
        for n in range(0, N, 7):
            for kb in range(D // 16):
                blk = xf[b, h, n, kb * 16:(kb + 1) * 16]
                sb = sf[oracle.sf_index(bh, (N + 127) // 128, n, kb, D // 16)]
                s = np.float32(oracle.e4m3_decode(int(sb))) * g
                codes = np.array([_nib(payload[b, h, n], kb * 16 + i) for i in range(16)])
                if s == 0:
                    assert np.all(codes == 0)
                    continue
                y = blk.astype(np.float32) * np.float32(1.0) / s
                deq = _dec_codes(codes)
                # nearest grid point of y (clipped at 6), within fp32 rounding of the reciprocal
                yc = np.clip(y, -6, 6)
                err = np.abs(yc - deq)
                nearest = np.min(np.abs(np.abs(yc)[:, None] - E2M1[None, :]), axis=1)
                assert np.all(err <= nearest + 1e-5 * np.maximum(1, np.abs(yc)))
                # the block scale keeps the block maximum within ~6 (E4M3 rounding of the scale)
                assert np.abs(blk).max() / s <= 6.0 * (1 + 2 ** -4) + 1e-6


def test_mxfp4_hand_worked(golden_dir):
    gold = json.load(open(os.path.join(golden_dir, "mxfp4_block.json")))
    B, H, N, D = gold["shape"]
    vals = np.array(gold["values_key_channel"], dtype=np.float32).reshape(B, H, N, D)
    v = _bits(vals.reshape(-1).tolist(), (B, H, N, D))
    payload_t, sf = oracle.quant_mxfp4_v(v, threads=1)
    assert payload_t.shape == (1, 1, D, 64)
    want = np.array(gold["codes_key_channel_padded"])
    for d in range(D):
        for n in range(128):
            assert _nib(payload_t[0, 0, d], n) == want[n, d], (d, n)
    for d in range(D):
        for kb in range(4):
            assert sf[(d % 32) * 16 + (d // 32) * 4 + kb] == gold["scale_bytes_channel_block"][d][kb]


def test_mxfp4_power_of_two_rule_and_transpose():
    _, _, v = wl.make_custom(1, 2, 300, 64, seed=9, kind="wide")
    payload_t, sf = oracle.quant_mxfp4_v(wl.bf16_bits(v))
    vf = v.float().numpy()
    B, H, N, D = vf.shape
    npad = 384
    for h in range(H):
        for d in range(0, D, 5):
            for kb in range(npad // 32):
                keys = np.arange(kb * 32, min(kb * 32 + 32, N))
                byte = sf[(h * 3 + kb // 4) * 512 + (d % 32) * 16 + (d // 32) * 4 + kb % 4]
                e = int(byte) - 127
                if keys.size == 0:
                    assert byte == 0
                    continue
                amax = np.abs(vf[0, h, keys, d]).max()
                if amax == 0:
                    assert byte == 0
                    continue
                assert amax <= 6 * 2.0 ** e < 2 * amax or e == -127
                codes = np.array([_nib(payload_t[0, h, d], n) for n in keys])
                deq = _dec_codes(codes) * 2.0 ** e
                y = vf[0, h, keys, d] / 2.0 ** e
                nearest = np.min(np.abs(np.abs(y)[:, None] - E2M1[None, :]), axis=1)
                assert np.all(np.abs(y - deq / 2.0 ** e) <= nearest + 1e-12)
            # padded keys are zero codes
            assert all(_nib(payload_t[0, h, d], n) == 0 for n in range(N, npad))
