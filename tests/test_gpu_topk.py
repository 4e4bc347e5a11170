"""dsa_topk on the GPU is bit-exact against the oracle's top-k of the same fp32 rows."""
import numpy as np
import pytest
import torch

import oracle
from dsa_sparse_attention_02_gb300 import _lib, inputs
from gpu_helpers import DEV, geometry_for_rows

pytestmark = pytest.mark.gpu


def _run(rows, lengths, k):
    lengths = np.asarray(lengths)
    g = geometry_for_rows(lengths)
    stride = int(-(-lengths.max() // 4) * 4)
    sc = np.full((len(lengths), stride), np.float32(7.0e30), dtype=np.float32)   # junk past each row
    for t, r in enumerate(rows):
        sc[t, : len(r)] = r
    scores = torch.from_numpy(sc).to(DEV)
    idx = torch.full((len(lengths), k), -7, dtype=torch.int32, device=DEV)
    ws = _lib.workspace(_lib.dsa_topk_workspace_size(g, k), DEV)
    _lib.dsa_topk(g, scores, k, idx, ws)
    assert _lib.dsa_get_error(ws) == 0
    got = idx.cpu().numpy()
    for t, r in enumerate(rows):
        exp = oracle.topk_row(np.asarray(r, dtype=np.float32).astype(np.float64), k)
        assert np.array_equal(got[t], exp), (t, len(r), k)


def test_random_rows_many_lengths():
    rng = np.random.default_rng(1)
    lengths = [1, 5, 63, 64, 65, 2047, 2048, 2049, 3000, 5000, 8192, 12345, 16384]
    rows = [rng.standard_normal(n).astype(np.float32) for n in lengths]
    _run(rows, lengths, 2048)
    _run(rows, lengths, 64)
    _run(rows, lengths, 1)


def test_exact_ties_and_signed_zero():
    rng = np.random.default_rng(2)
    rows = [
        inputs.tied_scores(rng, 1, 10000, k=2048)[0],
        rng.integers(-3, 4, size=9000).astype(np.float32),          # massive ties
        np.zeros(5000, dtype=np.float32),                           # all equal
        np.where(rng.random(6000) < 0.5, np.float32(0.0), np.float32(-0.0)),
        np.concatenate([np.full(3000, 2.5, np.float32), np.full(3000, -1.0, np.float32)]),
        rng.standard_normal(7000).astype(np.float32) * np.float32(1e-30),   # subnormal-range values
        np.concatenate([rng.standard_normal(4000).astype(np.float32) * 1e30,
                        np.float32([3.0e38, -3.0e38, 3.0, -3.0])]),
    ]
    _run(rows, [len(r) for r in rows], 2048)


def test_k_equal_to_and_just_below_row_length():
    rng = np.random.default_rng(3)
    rows = [rng.standard_normal(16384).astype(np.float32), rng.standard_normal(2048).astype(np.float32)]
    _run(rows, [16384, 2048], 2048)
    _run(rows[:1], [16384], 16384)
    _run(rows[:1], [16384], 16383)


def test_long_rows_two_level_with_ties():
    rng = np.random.default_rng(5)
    # the long-context top-k workload: 131072 scores ~N(0,1) with 1% injected exact ties,
    # including several copies of the k-th value
    rows = list(inputs.tied_scores(rng, 3, 131072, k=2048))
    rows += [rng.standard_normal(16385).astype(np.float32), rng.standard_normal(40000).astype(np.float32),
             rng.integers(0, 5, size=100000).astype(np.float32), rng.standard_normal(300).astype(np.float32)]
    _run(rows, [len(r) for r in rows], 2048)


def test_rows_longer_than_context_are_read_only_up_to_position():
    # multi-query requests: row t reads only s <= pos(t)
    rng = np.random.default_rng(6)
    L, nq, k = 3000, 4, 2048
    sc = rng.standard_normal((nq, L)).astype(np.float32)
    seq = torch.tensor([L], dtype=torch.int32, device=DEV)
    cu = torch.tensor([0, nq], dtype=torch.int32, device=DEV)
    bt = torch.zeros(1, (L + 63) // 64, dtype=torch.int32, device=DEV)
    g = _lib.Geometry(seq, cu, bt, num_pages=bt.shape[1], max_seq_len=L, T=nq)
    scores = torch.from_numpy(sc).to(DEV)
    idx = torch.empty(nq, k, dtype=torch.int32, device=DEV)
    ws = _lib.workspace(_lib.dsa_topk_workspace_size(g, k), DEV)
    _lib.dsa_topk(g, scores, k, idx, ws)
    got = idx.cpu().numpy()
    for j in range(nq):
        pos = L - nq + j
        exp = oracle.topk_row(sc[j, : pos + 1].astype(np.float64), k)
        assert np.array_equal(got[j], exp)


def test_long_rows_multi_level_merges():
    """Rows cut into many 16384-position chunks whose lists merge over two or three
    levels: 262144 and 300000 positions at k = 2048 (16 and 19 chunks, fan-in 8), and
    k = 4096 and 8192 (fan-in 4 and 2), next to short rows of the same call whose later
    chunks hold no valid entry (their merge groups carry fewer valid entries than k)."""
    rng = np.random.default_rng(7)
    rows = list(inputs.tied_scores(rng, 2, 262144, k=2048))
    rows += [rng.standard_normal(300000).astype(np.float32), rng.standard_normal(16484).astype(np.float32),
             rng.standard_normal(1000).astype(np.float32), rng.standard_normal(20000).astype(np.float32),
             rng.integers(0, 3, size=140000).astype(np.float32)]
    lengths = [len(r) for r in rows]
    _run(rows, lengths, 2048)
    _run(rows, lengths, 4096)
    _run(rows[2:5], lengths[2:5], 8192)
    _run(rows[:1], lengths[:1], 1)


def test_third_digit_and_whole_bin_paths():
    """Rows whose keys differ only in their lowest bits after a sign split, so the
    selection needs all three radix digits (the third re-uses the first digit's cleared
    histogram); rows where the threshold bin is taken whole after one or two digits; and
    the same through the chunk and merge levels of a long row."""
    rng = np.random.default_rng(11)
    one = np.float32(1.0)
    ulps = (np.arange(9000, dtype=np.int64) + np.int64(np.float32(1.0).view(np.int32))).astype(np.int32).view(np.float32)
    third = np.concatenate([np.full(3000, -1.0, np.float32), rng.permutation(ulps)])       # 1 + j ulp, j < 9000
    dup_low = np.concatenate([rng.permutation(ulps)[:6000], rng.permutation(ulps)[:6000]])  # every value twice
    whole1 = np.concatenate([np.full(2048, 4.0, np.float32), rng.uniform(0, 1, 6000).astype(np.float32)])
    whole2 = np.concatenate([np.full(1000, 8.0, np.float32), np.full(1048, 4.0 + 2 ** -10, np.float32),
                             np.full(3000, 4.0, np.float32), rng.uniform(0, 1, 3000).astype(np.float32)])
    rows = [third, dup_low, whole1, whole2, one + rng.permutation(ulps - one)]
    for k in (2048, 777, 1):
        _run(rows, [len(r) for r in rows], k)
    long_row = np.concatenate([rng.permutation(np.tile(ulps, 4)), np.full(5000, -2.0, np.float32)])
    _run([long_row], [len(long_row)], 2048)
    _run([long_row], [len(long_row)], 100)
