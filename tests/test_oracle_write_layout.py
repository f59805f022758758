"""Pins of the oracle's cache layouts and writer against what the pages print
(the fp8 K/V view shapes, the largest page id, the MXFP4 byte budget) and
against torch's e4m3 cast for the stored bytes."""
import os

import numpy as np
import pytest
import torch

import oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def geometry():
    g = {}
    for line in open(os.path.join(GOLD, "page_geometry.txt")):
        line = line.strip()
        if line and not line.startswith("#"):
            k, v = line.split()
            g[k] = tuple(int(x) for x in v.split(",")) if "," in v else int(v)
    return g


def bf16(x):
    return torch.tensor(np.asarray(x, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def f32(b):
    return O.bf16_to_f32(b)


def torch_e4m3(x):
    x = np.clip(np.asarray(x, np.float32), -448, 448)
    return torch.tensor(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def test_mxfp4_byte_budget():
    g = geometry()
    assert O.MX_FIELD_BYTES == g["mx_field_bytes"] == g["mx_data_bytes"] + g["mx_scale_bytes"]
    assert g["mx_data_bytes"] == 128 * 64 and g["mx_scale_bytes"] == 128 * 4
    assert O.kv_block_bytes(O.MXFP4, 1) // 128 == g["mx_kv_bytes_per_token"]
    assert O.index_field_bytes(O.MXFP4) // 128 == g["mx_index_bytes_per_token"]
    assert O.index_field_bytes(O.FP8) == 128 * 128 + 128 * 4


@pytest.mark.parametrize("nblk", [128, 512, 55673])
def test_fp8_views_match_printed_shapes(nblk):
    g = geometry()
    hkv = 1
    page = 2048
    total = nblk * O.kv_block_bytes(O.FP8, hkv)
    k_view = (total // (hkv * page), hkv, 8, 16, 16)
    v_view = ((total - 8 * page * hkv) // (hkv * page), hkv, 1, 128, 16)
    assert k_view == g[f"blocks_{nblk}_k_view"]
    assert v_view == g[f"blocks_{nblk}_v_view"]


def test_fp8_write_lands_where_the_views_say():
    """Write tokens with the oracle, then read them back through numpy
    reshapes to the printed K view [ids, Hkv, 8, 16, 16] and V view
    [ids-8, Hkv, 1, 128, 16]."""
    nblk, hkv = 6, 2
    rng = np.random.default_rng(0)
    kv = np.zeros(nblk * O.kv_block_bytes(O.FP8, hkv), np.uint8)
    T = 40
    slots = rng.choice(nblk * 128, T, replace=False).astype(np.int64)
    k = bf16(rng.standard_normal((T, hkv, 128)))
    v = bf16(rng.standard_normal((T, hkv, 128)))
    ks, vs = 0.0095, 0.0105
    O.kv_page_write(O.FP8, hkv, kv, ks, vs, O.FP8, hkv, np.zeros(nblk * hkv * 16896, np.uint8), k, v, None, slots)
    kview = kv.reshape(nblk * 16, hkv, 8, 16, 16)
    vview = kv[8 * 2048 * hkv:].reshape(nblk * 16 - 8, hkv, 1, 128, 16)
    for i, s in enumerate(slots):
        B, o = divmod(int(s), 128)
        P, t = B * 16 + o // 16, o % 16
        for h in range(hkv):
            ek = torch_e4m3(f32(k[i, h]) / np.float32(ks))
            ev = torch_e4m3(f32(v[i, h]) / np.float32(vs))
            got_k = np.array([kview[P, h, d // 16, t, d % 16] for d in range(128)])
            got_v = np.array([vview[P, h, 0, d, t] for d in range(128)])
            assert np.array_equal(got_k, ek) and np.array_equal(got_v, ev)


def test_bf16_write_is_a_copy_in_the_x8_layout():
    nblk, hkv = 2, 1
    kv = np.zeros(nblk * O.kv_block_bytes(O.BF16, hkv), np.uint8)
    rng = np.random.default_rng(1)
    k = bf16(rng.standard_normal((3, hkv, 128)))
    v = bf16(rng.standard_normal((3, hkv, 128)))
    slots = np.array([5, 130, 255], np.int64)
    O.kv_page_write(O.BF16, hkv, kv, 1.0, 1.0, O.BF16, hkv, np.zeros(nblk * 32768, np.uint8), k, v, None, slots)
    words = kv.view(np.uint16)
    kview = words.reshape(nblk * 16, hkv, 16, 16, 8)
    vview = words[8 * 2048 * hkv:].reshape(nblk * 16 - 8, hkv, 2, 128, 8)
    for i, s in enumerate(slots):
        B, o = divmod(int(s), 128)
        P, t = B * 16 + o // 16, o % 16
        assert np.array_equal(np.array([kview[P, 0, d // 8, t, d % 8] for d in range(128)]), k[i, 0])
        assert np.array_equal(np.array([vview[P, 0, t // 8, d, t % 8] for d in range(128)]), v[i, 0])


def test_mxfp4_write_field_layout_and_round_trip():
    nblk, hkv = 3, 2
    rng = np.random.default_rng(2)
    kv = np.zeros(nblk * O.kv_block_bytes(O.MXFP4, hkv), np.uint8)
    idx = np.zeros(nblk * hkv * O.MX_FIELD_BYTES, np.uint8)
    T = 20
    slots = rng.choice(nblk * 128, T, replace=False).astype(np.int64)
    # values on the e2m1 grid times a per-group power of two: exact round trip
    mags = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
    g = rng.choice(mags, (T, hkv, 4, 32)) * rng.choice([-1.0, 1.0], (T, hkv, 4, 32))
    g[..., 0] = 6.0
    g[..., 1] = 0.5
    ex = rng.integers(-5, 6, (T, hkv, 4, 1))
    x = (g * 2.0 ** ex).reshape(T, hkv, 128)
    k = bf16(x)
    v = bf16(-x)
    O.kv_page_write(O.MXFP4, hkv, kv, 1.0, 1.0, O.MXFP4, hkv, idx, k, v, k, slots)
    for i, s in enumerate(slots):
        B, o = divmod(int(s), 128)
        for h in range(hkv):
            for side, src in ((0, x), (1, -x)):
                base = O.mx_field_offset(hkv, B, side, h)
                assert base == B * 2 * hkv * 8704 + (side * hkv + h) * 8704
                fld = kv[base:base + 8704]
                for d in range(128):
                    byte = fld[o * 64 + d // 2]
                    nib = byte & 15 if d % 2 == 0 else byte >> 4
                    sc = fld[8192 + o * 4 + d // 32]
                    assert sc == ex[i, h, d // 32, 0] + 127
                    assert O.e2m1_decode(nib) * 2.0 ** (int(sc) - 127) == src[i, h, d]
            ifld = idx[(B * hkv + h) * 8704:(B * hkv + h + 1) * 8704]
            kfld = kv[O.mx_field_offset(hkv, B, 0, h):][:8704]
            assert np.array_equal(ifld[o * 64:(o + 1) * 64], kfld[o * 64:(o + 1) * 64])


def test_fp8_index_key_per_token_scale():
    nblk, hidx = 2, 1
    rng = np.random.default_rng(3)
    idx = np.zeros(nblk * hidx * 16896, np.uint8)
    kv = np.zeros(nblk * O.kv_block_bytes(O.FP8, 1), np.uint8)
    T = 10
    slots = rng.choice(nblk * 128, T, replace=False).astype(np.int64)
    x = rng.standard_normal((T, hidx, 128)) * rng.uniform(0.01, 100, (T, 1, 1))
    x[0] = 0.0
    ik = bf16(x)
    z = np.zeros((T, 1, 128), np.uint16)
    O.kv_page_write(O.FP8, 1, kv, 1.0, 1.0, O.FP8, hidx, idx, z, z, ik, slots)
    for i, s in enumerate(slots):
        B, o = divmod(int(s), 128)
        fld = idx[B * 16896:(B + 1) * 16896]
        xf = f32(ik[i, 0])
        amax = np.abs(xf).max()
        sc = np.float32(amax) / np.float32(448.0) if amax > 0 else np.float32(1.0)
        assert fld[16384 + 4 * o:16388 + 4 * o].view(np.float32)[0] == sc
        assert np.array_equal(fld[o * 128:(o + 1) * 128], torch_e4m3(xf / sc))


def test_skipped_slots_write_nothing():
    kv = np.zeros(O.kv_block_bytes(O.FP8, 1), np.uint8)
    idx = np.zeros(16896, np.uint8)
    k = bf16(np.ones((2, 1, 128)))
    O.kv_page_write(O.FP8, 1, kv, 0.5, 0.5, O.FP8, 1, idx, k, k, k, np.array([-1, -1], np.int64))
    assert not kv.any() and not idx.any()
