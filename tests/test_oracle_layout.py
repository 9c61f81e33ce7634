"""Pins of the oracle's own packer: the bytes of the packed weights and of the
activation workspace (buffer layout version 1) that the CUDA packer and the
CUDA activation kernel are compared with, byte for byte, on the GPU.

The oracle packer is checked against what fixes the layout independently of
its code: hand-derived byte positions of the layout statement
(tests/golden/layout_v1_positions.txt), the FP8 E4M3 format (torch's own
float8_e4m3fn cast), and invariants of a re-ordering (every input value lands
in exactly one place, the defined bytes fill each section exactly)."""
import os

import numpy as np
import pytest
import torch

import oracle

GOLD = os.path.join(os.path.dirname(__file__), "golden", "layout_v1_positions.txt")


def _golden():
    out = []
    for line in open(GOLD):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        kind, dims, idx, pos = (f.split() for f in line.split("|"))
        out.append((kind[0], [int(v) for v in dims], [int(v) for v in idx], [int(v) for v in pos]))
    return out


def test_e4m3_bytes_match_torch_float8_cast():
    codes = np.arange(-8, 9)
    ref = torch.tensor(codes, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert [oracle.e4m3_of_int(int(c)) for c in codes] == ref.tolist()


def _weights_probe(N, K, r, n, k):
    """Codes all 0 but one 7 at (n, k): nibble 8 everywhere except one 15."""
    qW = np.zeros((N, K), np.int8)
    qW[n, k] = 7
    sW = np.zeros((N, K // 64), np.uint16)
    Ld = np.zeros((K, r), np.uint16) if r else None
    Lu = np.zeros((r, N), np.uint16) if r else None
    return oracle.pack_weights_v1(qW, sW, Ld, Lu)


@pytest.mark.parametrize("entry", [e for e in _golden() if e[0] == "wcode"], ids=str)
def test_weight_code_positions_golden(entry):
    _, (N, K), (n, k), (byte, hi) = entry
    out, _ = _weights_probe(N, K, 0, n, k)
    sec = out[oracle.packed_offsets(N, K, 0)["qW"]:][: (K // 64) * N * 32]
    nib = np.stack([sec & 15, sec >> 4], axis=1)  # [byte, low/high]
    hits = np.argwhere(nib == 15)
    assert hits.tolist() == [[byte, hi]]
    assert (nib == 8).sum() == nib.size - 1


def _lora_probe(kind, dims, idx):
    if kind == "ld":
        K, r = dims
        N = 16
        Ld = np.zeros((K, r), np.uint16)
        Ld[idx[0], idx[1]] = 0x3C00  # 1.0
        Lu = np.zeros((r, N), np.uint16)
    else:
        N, r = dims
        K = 64
        Ld = np.zeros((K, r), np.uint16)
        Lu = np.zeros((r, N), np.uint16)
        Lu[idx[0], idx[1]] = 0x3C00
    out, _ = oracle.pack_weights_v1(np.zeros((N, K), np.int8), np.zeros((N, K // 64), np.uint16), Ld, Lu)
    off = oracle.packed_offsets(N, K, r)
    return out, off["Ld"] if kind == "ld" else off["Lu"]


@pytest.mark.parametrize("entry", [e for e in _golden() if e[0] in ("ld", "lu")], ids=str)
def test_lora_factor_positions_golden(entry):
    kind, dims, idx, (byte,) = entry
    out, base = _lora_probe(kind, dims, idx)
    nz = np.flatnonzero(out[base:] if kind == "lu" else out[:oracle.packed_offsets(16, dims[0], dims[1])["qW"]])
    # the fp16 value 1.0 = 0x3C00: only its high byte is nonzero
    assert nz.tolist() == [byte + 1]


def _act_probe(M, K, r, m, what, idx):
    qA = np.zeros((M, K), np.int8)
    sA = np.zeros((M, K // 64), np.float32)
    La = np.zeros((M, r), np.uint16) if r else None
    if what == "act":
        qA[m, idx] = 7
    elif what == "ss":
        sA[m, idx] = 1.0
    else:
        La[m, idx] = 0x3C00
    return oracle.pack_act_v1(qA, sA, La, r)


@pytest.mark.parametrize("entry", [e for e in _golden() if e[0] in ("act", "ss", "la")], ids=str)
def test_workspace_positions_golden(entry):
    kind, (M, d2), (m, i), (byte,) = entry
    K, r = (d2, 0) if kind in ("act", "ss") else (128, d2)
    out, _ = _act_probe(M, K, r, m, kind, i)
    off = oracle.act_offsets(M, K, r)
    if kind == "act":
        sec = out[off["qA"]:off["sS"]]
        assert np.flatnonzero(sec).tolist() == [byte]
        assert sec[byte] == 0x4E  # E4M3 of 7
    elif kind == "ss":
        sec = out[off["sS"]:off["La"]].view(np.float32)
        # sA = 1.0 at the probe; SA (the code sum) is 0 everywhere
        assert np.flatnonzero(sec).tolist() == [byte // 4]
    else:
        sec = out[off["La"]:off["flags"]]
        assert np.flatnonzero(sec).tolist() == [byte + 1]


def test_weight_packing_is_a_permutation():
    """Random codes, scales and LoRA factors: each value appears exactly once, and
    the defined bytes are exactly the sections' sizes; one-hot probes of all 64
    positions of a group land on 64 distinct nibbles of its record."""
    rng = np.random.default_rng(0)
    N, K, r = 48, 192, 32
    G = K // 64
    qW = rng.integers(-8, 8, (N, K)).astype(np.int8)
    sW = rng.integers(0, 1 << 15, (N, G)).astype(np.uint16)
    Ld = np.arange(K * r, dtype=np.uint16).reshape(K, r)          # all distinct
    Lu = (np.arange(r * N, dtype=np.uint16) + 40000).reshape(r, N)
    out, defined = oracle.pack_weights_v1(qW, sW, Ld, Lu)
    off = oracle.packed_offsets(N, K, r)
    assert defined.sum() == K * r * 2 + G * N * 32 + G * N * 2 + r * N * 2
    sec = out[off["qW"]:off["qW"] + G * N * 32]
    nibs = np.concatenate([sec & 15, sec >> 4]).astype(np.int64) - 8
    assert np.array_equal(np.bincount(nibs + 8, minlength=16), np.bincount(qW.ravel().astype(np.int64) + 8, minlength=16))
    # every record holds exactly the 64 codes of its (group, row)
    rec = sec.reshape(G, N, 32)
    for g in range(G):
        for n in (0, 7, N - 1):
            got = np.sort(np.concatenate([rec[g, n] & 15, rec[g, n] >> 4]).astype(np.int64) - 8)
            assert np.array_equal(got, np.sort(qW[n, 64 * g:64 * g + 64].astype(np.int64)))
    ld = out[off["Ld"]:off["Ld"] + K * r * 2].view(np.uint16)
    assert np.array_equal(np.sort(ld), np.sort(Ld.ravel()))
    sw = out[off["sW"]:off["sW"] + G * N * 2].view(np.uint16).reshape(G, N)
    assert np.array_equal(sw, sW.T)  # [G][N], unswizzled
    lu = out[off["Lu"]:off["Lu"] + r * N * 2].view(np.uint16)
    assert np.array_equal(np.sort(lu), np.sort(Lu.ravel()))
    seen = set()
    for k in range(64):
        o, _ = _weights_probe(16, 64, 0, 2, k)
        rec2 = o[oracle.packed_offsets(16, 64, 0)["qW"] + 2 * 32:][:32]
        nib = np.stack([rec2 & 15, rec2 >> 4], axis=1)
        (pos,) = [tuple(p) for p in np.argwhere(nib == 15)]
        seen.add(pos)
    assert len(seen) == 64


def test_workspace_packing_is_a_permutation():
    rng = np.random.default_rng(1)
    M, K, r = 300, 192, 32
    G = K // 64
    qA = rng.integers(-8, 8, (M, K)).astype(np.int8)
    sA = rng.uniform(0.01, 1.0, (M, G)).astype(np.float32)
    La = rng.integers(0, 1 << 15, (M, r)).astype(np.uint16)
    out, defined = oracle.pack_act_v1(qA, sA, La, r)
    off = oracle.act_offsets(M, K, r)
    assert defined.sum() == M * K + M * G * 8 + M * r * 2 + 160 * 16 * 4
    e4m3 = {c: oracle.e4m3_of_int(c) for c in range(-8, 8)}
    codes = out[off["qA"]:off["sS"]][defined[off["qA"]:off["sS"]] == 1]
    want = np.array([e4m3[int(c)] for c in qA.ravel()], np.uint8)
    assert np.array_equal(np.sort(codes), np.sort(want))
    ss = out[off["sS"]:off["La"]].view(np.float32).reshape(-1, 128, 2)  # [MT * G][128][2]
    MT = (M + 127) // 128
    ss = ss.reshape(MT, G, 128, 2)
    for m in (0, 5, 127, 128, M - 1):
        for g in range(G):
            assert ss[m // 128, g, m % 128, 0] == sA[m, g]
            assert ss[m // 128, g, m % 128, 1] == float(qA[m, 64 * g:64 * g + 64].astype(np.int64).sum())
    la = out[off["La"]:off["flags"]][defined[off["La"]:off["flags"]] == 1].view(np.uint16)
    assert np.array_equal(np.sort(la), np.sort(La.ravel()))
    assert not out[off["flags"]:off["total"]].any() and defined[off["flags"]:off["total"]].all()
