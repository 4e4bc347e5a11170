"""The seeded synthetic workloads have the shapes and structure the configurations state."""
import numpy as np
import pytest

from dsa_sparse_attention_02_gb300 import inputs as synth


def _check_geometry(wl):
    pages = (wl.seq_lens.astype(np.int64) + 63) // 64
    used = np.concatenate([wl.block_table[b, :pages[b]] for b in range(wl.B)])
    assert len(np.unique(used)) == len(used)                 # no page shared
    assert used.min() >= 0 and used.max() < wl.num_pages
    assert wl.num_pages >= pages.sum()                        # spare pages exist
    assert wl.cu_q[0] == 0 and np.all(np.diff(wl.cu_q) == wl.n_q)


def test_tiny_config_shapes():
    wl = synth.make_config("tiny")
    _check_geometry(wl)
    assert wl.seq_lens.tolist() == [200, 256] and wl.T == 2 and wl.topk == 64
    assert wl.q_idx.shape == (2, 4, 128) and wl.q_idx.dtype == np.uint16
    assert wl.idx_k_scale is None and wl.qk_dtype == "bf16"
    assert wl.layers[0].q.shape == (2, 16, 576) and wl.layers[0].kv.shape[1:] == (64, 576)
    assert abs(wl.sm_scale - 192 ** -0.5) < 1e-15


def test_small_variants_of_large_configs():
    wl = synth.make_config("decode", batch=4)
    _check_geometry(wl)
    assert np.all((wl.seq_lens >= 2048) & (wl.seq_lens <= 8192))
    assert wl.q_idx.dtype == np.uint8 and wl.q_scale.shape == (4, 64)
    wl = synth.make_config("mtp", batch=2, ctx_scale=0.25)
    _check_geometry(wl)
    assert wl.T == 8 and len(wl.layers) == 2 and wl.layers[0].kv.shape[-1] == 64 * 656
    wl = synth.make_config("longctx", batch=1, ctx_scale=1 / 64)
    _check_geometry(wl)
    assert wl.seq_lens.tolist() == [2048]


def test_seeded_and_reproducible():
    a = synth.make_config("decode", batch=3)
    b = synth.make_config("decode", batch=3)
    assert np.array_equal(a.idx_k, b.idx_k) and np.array_equal(a.layers[0].kv, b.layers[0].kv)


def test_duplicated_index_keys_tie():
    wl = synth.make_config("longctx", batch=1, ctx_scale=1 / 32)
    flat = wl.idx_k.reshape(-1, 128)
    rows = wl.block_table[0, :64].astype(np.int64)[:, None] * 64 + np.arange(64)[None]
    keys = flat[rows.reshape(-1)[: wl.seq_lens[0]]]
    uniq = np.unique(keys, axis=0)
    assert len(uniq) < len(keys)


def test_fp8_quantization_saturates_and_rounds():
    codes, scale = synth.quantize_rows_e4m3(np.array([[448.0, -1000.0, 1.0, 0.0]], np.float32), 4)
    assert scale[0, 0] == np.float32(1000.0 / 448.0)
    assert codes[0, 1] == 0xFE                                 # -448, not NaN
    assert synth.to_e4m3_bytes(np.array([449.0, 500.0], np.float32)).tolist() == [0x7E, 0x7E]


def test_tied_score_rows():
    rng = np.random.default_rng(0)
    s = synth.tied_scores(rng, 2, 10000, k=2048)
    for r in range(2):
        kth = np.sort(s[r])[::-1][2047]
        assert (s[r] == kth).sum() >= 2
