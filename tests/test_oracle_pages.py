"""Pins of the oracle's page writer against the documented page layout.

Section sizes are checked against hand-computed byte counts; packed rows are
unpacked with numpy.unpackbits (little bit order) and compared with the codes.
"""
import numpy as np
import pytest

import kvq_inputs as W
from oracle import kvq_oracle as O


def test_layout_config5_by_hand():
    # INT8 sym K per-channel G=64, INT4 asym V per-token g=128, P=16, D=128, Hkv=8
    cfg = O.Config(32, 8, 128, O.QSpec(O.INT8, O.SYM, O.PER_CHANNEL, 64),
                   O.QSpec(O.INT4, O.ASYM, O.PER_TOKEN, 128), residual=64, page_size=16)
    L = O.layout(cfg)
    # K codes 16*128 = 2048, V codes 16*64 = 1024, V meta 16*(1 scale + 1 min)*4 = 128,
    # K meta max(1, 16/64) = 1 group * 128 scales * 4 = 512
    assert (L["kc"], L["vc"], L["vm"], L["km"], L["head"]) == (0, 2048, 3072, 3200, 3712)
    assert L["page"] == 8 * 3712


def test_layout_config3_by_hand():
    # INT2 asym K per-channel G=32, INT2 asym V per-token g=32, P=256
    cfg = O.Config(32, 8, 128, O.QSpec(O.INT2, O.ASYM, O.PER_CHANNEL, 32),
                   O.QSpec(O.INT2, O.ASYM, O.PER_TOKEN, 32), residual=128, page_size=256)
    L = O.layout(cfg)
    # K codes 256*32 = 8192; V codes 8192; V meta 256 * 4 groups * 2 * 4 = 8192;
    # K meta 8 groups * 128 * 2 * 4 = 8192
    assert (L["kc"], L["vc"], L["vm"], L["km"], L["head"]) == (0, 8192, 16384, 24576, 32768)


def _unpack(row_bytes, bits, D):
    bitsarr = np.unpackbits(np.asarray(row_bytes, np.uint8), bitorder="little")
    w = 2 ** np.arange(bits)
    return (bitsarr[:D * bits].reshape(D, bits) * w).sum(axis=1)


@pytest.mark.parametrize("kfmt,kmode,vfmt,vmode", [
    (O.INT2, O.ASYM, O.INT2, O.ASYM), (O.INT4, O.SYM, O.INT4, O.ASYM), (O.INT8, O.SYM, O.INT2, O.SYM),
    (O.INT8, O.ASYM, O.INT8, O.SYM)])
def test_page_writer_roundtrip(kfmt, kmode, vfmt, vmode):
    D, P, G, R = 64, 16, 32, 64
    cfg = O.Config(2, 2, D, O.QSpec(kfmt, kmode, O.PER_CHANNEL, G), O.QSpec(vfmt, vmode, O.PER_TOKEN, 32),
                   residual=R, page_size=P)
    L = O.layout(cfg)
    T = 150
    n_pages = 40
    bt = np.array([np.arange(20) * 2, np.arange(20) * 2 + 1], dtype=np.int32)
    pages = np.zeros((n_pages, L["page"]), np.uint8)
    defined = np.zeros_like(pages, dtype=bool)
    states = {}
    for b in range(2):
        for h in range(2):
            K = W.small_stream(10 + b * 2 + h, T, D, (4,), 25.0)
            V = W.small_stream(20 + b * 2 + h, T, D)
            st = O.quantize_stream(cfg, K, V)
            states[b, h] = st
            O.write_head_pages(cfg, pages, defined, bt, b, h, st)
    kb, vb = O.bits_of(kfmt), O.bits_of(vfmt)
    for (b, h), st in states.items():
        assert st.n_q == 128
        for t in range(st.n_q):
            page, slot = bt[b][t // P], t % P
            base = h * L["head"]
            krow = pages[page, base + slot * L["krow"]: base + (slot + 1) * L["krow"]]
            u = _unpack(krow, kb, D)
            want = st.kc[t]
            want = want + (2 ** (kb - 1) if (kmode == O.SYM and kb < 8) else 0)
            want = np.where(want < 0, want + 256, want)
            assert np.array_equal(u, want)
            vrow = pages[page, base + L["vc"] + slot * L["vrow"]: base + L["vc"] + (slot + 1) * L["vrow"]]
            w = st.vc[t] + (2 ** (vb - 1) if (vmode == O.SYM and vb < 8) else 0)
            assert np.array_equal(_unpack(vrow, vb, D), np.where(w < 0, w + 256, w))
            nm = 2 if vmode == O.ASYM else 1
            meta = pages[page, base + L["vm"] + slot * 2 * nm * 4: base + L["vm"] + (slot + 1) * 2 * nm * 4]
            mf = meta.view(np.float32)
            assert np.array_equal(mf[:2], st.vs[t].astype(np.float32))
            if nm == 2:
                assert np.array_equal(mf[2:], st.vm[t].astype(np.float32))
        for j in range(st.n_q // G):
            page = bt[b][(j * G) // P]
            base = h * L["head"] + L["km"]
            nm = 2 if kmode == O.ASYM else 1
            mf = pages[page, base: base + D * nm * 4].view(np.float32)
            assert np.array_equal(mf[:D], st.ks[j].astype(np.float32))
            if nm == 2:
                assert np.array_equal(mf[D:], st.km[j].astype(np.float32))
    # pages never touched stay undefined; every defined byte belongs to a used page
    used = {int(bt[b][t // P]) for b in range(2) for t in range(128)}
    assert set(np.nonzero(defined.any(axis=1))[0].tolist()) == used


# Per-token keys and binary16 metadata, worked by hand on a 4-token page, D = 8.
# K: asymmetric INT4 per token in two groups of 4 channels; V: symmetric INT8 per
# token (one group).  Every scale is exact (ranges 15 and absmax 127).
#   K row 0: [0, 15, 1, 2 | -8, 7, 0, 1]  -> group 0: min 0, s 1, codes 0 15 1 2
#                                            group 1: min -8, s 1, codes 0 15 8 9
#   packed little-endian, low nibble first: F0 21 F0 98
#   K row 1: [3, 3, 3, 3 | 1, 16, 2, 3]   -> group 0 constant: d = 1e-8 (fl32), codes 0 0 0 0,
#                                            min 3; group 1: min 1, s 1, codes 0 15 1 2
#   packed: 00 00 F0 21
#   V row 0: [127, -127, 1, 0.5, 2.5, -1.5, 0, 64] -> s 1, codes 127 -127 1 0 2 -2 0 64
#   bytes (two's complement): 7F 81 01 00 02 FE 00 40
#   V row 1: [-127, 0, 0, 0, 0, 0, 0, 3.5]  -> s 1, codes -127 0 0 0 0 0 0 4: 81 00 00 00 00 00 00 04
# Section offsets (16-byte aligned, in the order K codes, V codes, V meta, K meta):
#   fp32 meta: K codes 4 x 4 = 16 at 0; V codes 4 x 8 = 32 at 16; V meta 4 x 1 x 4 = 16 at 48;
#              K meta 4 tokens x (2 scales + 2 minima) x 4 = 64 at 64; head block 128
#   binary16:  V meta 4 x 2 = 8 at 48; K meta 4 x 4 x 2 = 32 at 64 (48 + 8 rounded up); head 96
_HAND_K = [[0, 15, 1, 2, -8, 7, 0, 1], [3, 3, 3, 3, 1, 16, 2, 3]]
_HAND_V = [[127, -127, 1, 0.5, 2.5, -1.5, 0, 64], [-127, 0, 0, 0, 0, 0, 0, 3.5]]


def _hand_cfg(meta):
    return O.Config(1, 1, 8, O.QSpec(O.INT4, O.ASYM, O.PER_TOKEN, 4), O.QSpec(O.INT8, O.SYM, O.PER_TOKEN, 8),
                    residual=0, page_size=4, meta_dtype=meta)


@pytest.mark.parametrize("meta", [O.F32, O.F16])
def test_per_token_key_pages_by_hand(meta):
    cfg = _hand_cfg(meta)
    L = O.layout(cfg)
    want_layout = (0, 16, 48, 64, 128) if meta == O.F32 else (0, 16, 48, 64, 96)
    assert (L["kc"], L["vc"], L["vm"], L["km"], L["head"]) == want_layout
    st = O.quantize_stream(cfg, np.array(_HAND_K, float), np.array(_HAND_V, float))
    pages = np.zeros((3, L["page"]), np.uint8)
    defined = np.zeros_like(pages, dtype=bool)
    O.write_head_pages(cfg, pages, defined, np.array([[2]], np.int32), 0, 0, st)
    pg = pages[2]
    assert pg[0:8].tolist() == [0xF0, 0x21, 0xF0, 0x98, 0x00, 0x00, 0xF0, 0x21]
    assert pg[16:32].tolist() == [0x7F, 0x81, 0x01, 0x00, 0x02, 0xFE, 0x00, 0x40,
                                  0x81, 0x00, 0x00, 0x00, 0x00, 0x00, 0x00, 0x04]
    tiny = float(np.float32(1e-8) / np.float32(15))  # constant group: max(d, 1e-8) / qmax in fp32
    if meta == O.F32:
        # V meta: one fp32 scale per token; K meta: per token (scale g0, scale g1, min g0, min g1)
        assert pg[48:56].tolist() == [0, 0, 0x80, 0x3F] * 2  # 1.0f
        assert pg[64:72].tolist() == [0, 0, 0x80, 0x3F, 0, 0, 0x80, 0x3F]  # 1.0f, 1.0f
        assert pg[72:80].tolist() == [0, 0, 0, 0, 0, 0, 0, 0xC1]  # 0.0f, -8.0f
        row1 = pg[80:96].view(np.float32)
        assert row1[0] == np.float32(tiny) and row1[1] == 1.0 and row1[2] == 3.0 and row1[3] == 1.0
        assert not defined[2, 96:128].any()  # the two unused slots stay undefined
    else:
        # binary16: 1.0 = 0x3C00, -8.0 = 0xC800, 3.0 = 0x4200, little-endian; the constant
        # group's tiny scale rounds up to the smallest subnormal half (2^-24 = 0x0001)
        assert pg[48:52].tolist() == [0x00, 0x3C, 0x00, 0x3C]
        assert pg[64:72].tolist() == [0x00, 0x3C, 0x00, 0x3C, 0x00, 0x00, 0x00, 0xC8]
        assert pg[72:80].tolist() == [0x01, 0x00, 0x00, 0x3C, 0x00, 0x42, 0x00, 0x3C]
        assert not defined[2, 80:96].any()
    assert not defined[0].any() and not defined[1].any()
