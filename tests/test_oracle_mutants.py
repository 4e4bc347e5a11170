"""Planted mistakes in the CPU oracle, on the CPU: each case edits one function of
`oracle/` in memory (a dropped term, a wrong sign, index or bound, a swapped operand,
a wrong constant or rounding rule), rebinds it wherever the oracle refers to it, and
runs every pin of the oracle (test_oracle_pins, test_oracle_cache, test_oracle_prep)
against the edited oracle. At least one pin must fail for every planted mistake;
a mistake that no pin notices is a hole in the pins.

Each edit names the exact source text it replaces, so a change to the oracle that
moves that text fails here loudly instead of silently testing nothing.
"""
import contextlib
import inspect
import itertools
import sys
import textwrap
import warnings

import numpy as np
import pytest

import oracle
import oracle.cache
import oracle.dsa
import oracle.fp8
import oracle.prep

import test_oracle_cache
import test_oracle_pins
import test_oracle_prep

PIN_MODULES = (test_oracle_pins, test_oracle_cache, test_oracle_prep)

# (case id, oracle module, function, [(old source text, new source text), ...])
MUTANTS = [
    # storage formats
    ("e4m3-bias-8", "fp8", "_e4m3_value", [("2.0 ** (exp - 7)", "2.0 ** (exp - 8)")]),
    ("e4m3-subnormal-implicit-one", "fp8", "_e4m3_value",
     [("return sign * man * 2.0 ** -9", "return sign * (1.0 + man / 8.0) * 2.0 ** -6")]),
    ("e4m3-nan-whole-top-binade", "fp8", "_e4m3_value", [("if exp == 0xF and man == 0x7:", "if exp == 0xF:")]),
    ("bf16-read-as-fp16", "fp8", "decode_bf16",
     [("return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)",
       "return bits.view(np.float16).astype(np.float64)")]),
    ("int8-read-unsigned", "fp8", "decode_int8", [("codes.view(np.int8)", "codes.view(np.uint8)")]),
    ("f32-big-endian", "fp8", "decode_f32le", [('"<f4"', '">f4"')]),
    # geometry
    ("position-off-by-one", "dsa", "query_positions", [("pos.append(L - n + j)", "pos.append(L - n + j + 1)")]),
    ("positions-reversed", "dsa", "query_positions", [("pos.append(L - n + j)", "pos.append(L - 1 - j)")]),
    ("page-id-not-scaled", "dsa", "physical_rows", [("[s // PAGE] * PAGE + s % PAGE", "[s // PAGE] + s % PAGE")]),
    ("page-and-offset-swapped", "dsa", "physical_rows",
     [("[s // PAGE] * PAGE + s % PAGE", "[s % PAGE] * PAGE + s // PAGE")]),
    # indexer operands
    ("q-scale-dropped", "dsa", "decode_index_q",
     [("return decode_e4m3(q_idx) * np.asarray(q_scale, dtype=np.float64)[..., None]",
       "return decode_e4m3(q_idx)")]),
    ("k-scale-dropped", "dsa", "decode_index_keys",
     [("return decode_e4m3(flat) * np.asarray(idx_k_scale, dtype=np.float64).reshape(-1)[rows][:, None]",
       "return decode_e4m3(flat)")]),
    ("k-scale-of-page-first-row", "dsa", "decode_index_keys",
     [(".reshape(-1)[rows][:, None]", ".reshape(-1)[np.asarray(rows) - np.asarray(rows) % 64][:, None]")]),
    ("latent-scales-interleaved", "dsa", "decode_kv_rows",
     [("np.repeat(scales, 128, axis=1)", "np.tile(scales, (1, 128))")]),
    ("rope-of-the-next-slot", "dsa", "decode_kv_rows",
     [("rope_bytes[page, slot]", "rope_bytes[page, (slot + 1) % PAGE]")]),
    ("int8-latent-decoded-as-e4m3", "dsa", "decode_kv_rows",
     [('if kv_dtype == "e4m3" else', 'if kv_dtype in ("e4m3", "int8") else')]),
    # indexer
    ("relu-dropped", "dsa", "indexer_scores", [("np.maximum(logits, 0.0) @", "logits @")]),
    ("relu-after-head-sum", "dsa", "indexer_scores",
     [("out[t] = np.maximum(logits, 0.0) @ np.asarray(w[t], dtype=np.float64)",
       "out[t] = np.maximum(logits @ np.asarray(w[t], dtype=np.float64), 0.0)")]),
    ("own-key-not-visible", "dsa", "indexer_scores", [("keys = cache[b][: p + 1]", "keys = cache[b][:p]")]),
    ("one-key-past-the-query", "dsa", "indexer_scores", [("keys = cache[b][: p + 1]", "keys = cache[b][: p + 2]")]),
    ("weights-of-first-token", "dsa", "indexer_scores",
     [("np.asarray(w[t], dtype=np.float64)", "np.asarray(w[0], dtype=np.float64)")]),
    ("head-weights-reversed", "dsa", "indexer_scores",
     [("np.asarray(w[t], dtype=np.float64)", "np.asarray(w[t][::-1], dtype=np.float64)")]),
    ("query-of-first-token", "dsa", "indexer_scores", [("q_idx[t:t + 1]", "q_idx[0:1]")]),
    ("keys-of-first-request", "dsa", "indexer_scores", [("if b not in cache:", "if not cache:")]),
    # top-k
    ("ties-to-higher-position", "dsa", "topk_row",
     [("np.lexsort((np.arange(n), -scores))", "np.lexsort((-np.arange(n), -scores))")]),
    ("smallest-k", "dsa", "topk_row", [("np.lexsort((np.arange(n), -scores))", "np.lexsort((np.arange(n), scores))")]),
    ("score-order-output", "dsa", "topk_row", [("keep = np.sort(order[: min(k, n)])", "keep = order[: min(k, n)]")]),
    ("padding-zero", "dsa", "topk_row", [("np.full(k, -1, dtype=np.int32)", "np.zeros(k, dtype=np.int32)")]),
    ("keeps-one-fewer", "dsa", "topk_row", [("order[: min(k, n)]", "order[: min(k, n) - 1]")]),
    # attention
    ("sm-scale-dropped", "dsa", "sparse_mla", [("z = sm_scale * (qt @ kvr.T)", "z = qt @ kvr.T")]),
    ("lse-without-max", "dsa", "sparse_mla", [("(m + np.log(l))[:, 0]", "np.log(l)[:, 0]")]),
    ("padding-attended", "dsa", "sparse_mla", [("sel = sel[sel >= 0]", "sel = sel.copy()")]),
    ("softmax-over-heads", "dsa", "sparse_mla",
     [("m = z.max(axis=1, keepdims=True)", "m = z.max(axis=0, keepdims=True)"),
      ("l = e.sum(axis=1, keepdims=True)", "l = e.sum(axis=0, keepdims=True)")]),
    ("values-from-the-tail", "dsa", "sparse_mla", [("kvr[:, :dv]", "kvr[:, -dv:]")]),
    ("empty-selection-lse-zero", "dsa", "sparse_mla", [("np.full(H, -np.inf)", "np.zeros(H)")]),
    ("empty-selection-output-nan", "dsa", "sparse_mla", [("np.zeros((H, dv))", "np.full((H, dv), np.nan)")]),
    # the step
    ("reused-selection-ignored", "dsa", "dsa_step", [("if reuse_idx is None:", "if True:")]),
    ("later-layer-own-queries-first-layer-cache", "dsa", "dsa_step", [("layer.kv, layer.kv_dtype", "wl.layers[0].kv, wl.layers[0].kv_dtype")]),
    # e4m3 / int8 encoders and the cache append
    ("e4m3-ties-away-from-zero", "cache", "encode_e4m3",
     [("((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))", "(d_hi == d_lo)")]),
    ("e4m3-ties-to-odd", "cache", "encode_e4m3",
     [("((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))", "((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 1))")]),
    ("e4m3-overflow-to-nan", "cache", "encode_e4m3",
     [("np.where(mag >= E4M3_MAX, np.uint8(0x7E), code)", "np.where(mag > E4M3_MAX, np.uint8(0x7F), code)")]),
    ("e4m3-negative-zero-positive", "cache", "encode_e4m3", [("neg = np.signbit(v)", "neg = v < 0")]),
    ("e4m3-scale-over-127", "cache", "group_scale", [("amax / np.float32(E4M3_MAX)", "amax / np.float32(127.0)")]),
    ("e4m3-amax-signed", "cache", "group_scale", [("amax = np.abs(x32).max(axis=-1)", "amax = x32.max(axis=-1)")]),
    ("int8-amax-signed", "cache", "quantize_groups_int8", [("amax = np.abs(g).max(axis=-1)", "amax = g.max(axis=-1)")]),
    ("e4m3-zero-group-scale-zero", "cache", "group_scale",
     [("np.float32(1.0)).astype(np.float32)", "np.float32(0.0)).astype(np.float32)")]),
    ("e4m3-quotient-in-float64", "cache", "quantize_groups",
     [("q = (g / scale[..., None]).astype(np.float32)",
       "q = g.astype(np.float64) / scale[..., None].astype(np.float64)")]),
    ("int8-ties-away-from-zero", "cache", "encode_int8",
     [("((frac == 0.5) & (np.mod(fl, 2) == 1))", "(frac == 0.5)")]),
    ("int8-clamp-at-minus-128", "cache", "encode_int8",
     [("np.clip(fl + up, -I8_MAX, I8_MAX)", "np.clip(fl + up, -I8_MAX - 1, I8_MAX)")]),
    ("int8-scale-over-448", "cache", "quantize_groups_int8",
     [("amax / np.float32(I8_MAX)", "amax / np.float32(E4M3_MAX)")]),
    ("append-position-off-by-one", "cache", "token_rows",
     [("pos = int(L) - int(n) + j", "pos = int(L) - int(n) + j + 1")]),
    ("append-rope-over-the-scales", "cache", "cache_append",
     [("rope_plane[page, slot] = np.ascontiguousarray", "scale_plane[page, slot, :] = 0\n"
       "            rope_plane[page, slot] = np.ascontiguousarray")]),
    ("record-rope-plane-offset", "dsa", "record_planes",
     [("pages[:, REC_ROPE_AT:].reshape", "pages[:, REC_ROPE_AT - 128:-128].reshape")]),
    ("record-scale-plane-not-per-token", "dsa", "record_planes",
     [("pages[:, REC_SCALES_AT:REC_ROPE_AT].reshape(P, PAGE, 16)",
       "pages[:, REC_SCALES_AT:REC_ROPE_AT].reshape(P, 16, PAGE).transpose(0, 2, 1)")]),
    ("append-key-scale-not-written", "cache", "cache_append", [("out_s[r] = scale[0]", "pass")]),
    ("append-e4m3-scale-per-row", "cache", "cache_append",
     [("codes, scales = quant(x[t, :512], 128)", "codes, scales = quant(x[t, :512], 512)\n"
       "            scales = np.repeat(scales, 4)")]),
    # indexer preparation
    ("rope-pairs-interleaved", "prep", "rope_rotate_half",
     [("a, b = x[..., :r], x[..., r:rope_dim]", "a, b = x[..., 0:rope_dim:2], x[..., 1:rope_dim:2]")]),
    ("rope-first-half-sign", "prep", "rope_rotate_half", [("y[..., :r] = a * c - b * s", "y[..., :r] = a * c + b * s")]),
    ("rope-second-half-sign", "prep", "rope_rotate_half",
     [("y[..., r:rope_dim] = b * c + a * s", "y[..., r:rope_dim] = b * c - a * s")]),
    ("rope-sin-cos-swapped", "prep", "rope_rotate_half",
     [("c, s = np.asarray(cos, dtype=np.float64), np.asarray(sin, dtype=np.float64)",
       "s, c = np.asarray(cos, dtype=np.float64), np.asarray(sin, dtype=np.float64)")]),
    ("layernorm-unbiased-variance", "prep", "layer_norm",
     [("((x - mu) ** 2).mean(axis=-1, keepdims=True)", "((x - mu) ** 2).sum(axis=-1, keepdims=True) / (x.shape[-1] - 1)")]),
    ("layernorm-eps-outside-sqrt", "prep", "layer_norm", [("np.sqrt(var + float(eps))", "(np.sqrt(var) + float(eps))")]),
    ("layernorm-beta-dropped", "prep", "layer_norm",
     [("* np.asarray(gamma, np.float64) + np.asarray(beta, np.float64)", "* np.asarray(gamma, np.float64)")]),
    ("layernorm-not-centred", "prep", "layer_norm", [("return (x - mu) /", "return x /")]),
    ("key-rope-before-layernorm", "prep", "prepared_k",
     [("kn = layer_norm(k, gamma, beta, eps)", "kn = k"),
      ("return rope_rotate_half(kn, c, s, rope_dim)",
       "return layer_norm(rope_rotate_half(kn, c, s, rope_dim), gamma, beta, eps)")]),
    ("key-not-normalized", "prep", "prepared_k", [("kn = layer_norm(k, gamma, beta, eps)", "kn = k")]),
    ("query-rope-one-position-late", "prep", "prepared_q",
     [("np.asarray(cos_table, np.float64)[pos]", "np.asarray(cos_table, np.float64)[pos + 1]"),
      ("np.asarray(sin_table, np.float64)[pos]", "np.asarray(sin_table, np.float64)[pos + 1]")]),
    ("query-scale-per-token", "prep", "indexer_prepare",
     [("quantize_groups(qx.astype(np.float32).reshape(T, H * DIM), DIM)",
       "quantize_groups(qx.astype(np.float32).reshape(T, H * DIM), H * DIM)\n"
       "    q_scale = np.repeat(q_scale, H, axis=1)")]),
    ("key-row-of-first-token", "prep", "indexer_prepare", [("kflat[r] = k_codes[t]", "kflat[r] = k_codes[0]")]),
]


def _oracle_modules():
    return [m for name, m in sys.modules.items() if name == "oracle" or name.startswith("oracle.")]


def _mutated(module, func, edits):
    """The function `func` of oracle.<module> compiled from its source with `edits`."""
    mod = getattr(oracle, module)
    orig = getattr(mod, func)
    src = textwrap.dedent(inspect.getsource(orig))
    for old, new in edits:
        assert src.count(old) == 1, f"{module}.{func}: expected exactly one {old!r} in its source"
        src = src.replace(old, new)
    ns = dict(mod.__dict__)
    exec(compile(src, f"<mutant of oracle.{module}.{func}>", "exec"), ns)
    return orig, ns[func]


@contextlib.contextmanager
def _planted(module, func, edits):
    """Rebinds every oracle reference to the original function (and, for the e4m3 value
    function, to the table built from it) to the mutant for the duration."""
    orig, new = _mutated(module, func, edits)
    swaps = [(orig, new)]
    if func == "_e4m3_value":
        table = np.array([new(c) for c in range(256)], dtype=np.float64)
        swaps.append((oracle.fp8.E4M3_TABLE, table))
    undo = []
    for m in _oracle_modules():
        for name, val in list(vars(m).items()):
            for o, n in swaps:
                if val is o:
                    undo.append((m, name, val))
                    setattr(m, name, n)
    try:
        yield
    finally:
        for m, name, val in undo:
            setattr(m, name, val)


def _pin_calls():
    """Every pin as (name, zero-argument callable), parametrized pins expanded."""
    calls = []
    for mod in PIN_MODULES:
        for name, f in sorted(vars(mod).items()):
            if not (name.startswith("test_") and callable(f)):
                continue
            marks = [m for m in getattr(f, "pytestmark", []) if m.name == "parametrize"]
            if not marks:
                calls.append((f"{mod.__name__}::{name}", f))
                continue
            combos = [[]]
            for m in marks:
                names = [a.strip() for a in m.args[0].split(",")] if isinstance(m.args[0], str) else list(m.args[0])
                vals = [v if len(names) > 1 else (v,) for v in m.args[1]]
                combos = [c + list(zip(names, v)) for c in combos for v in vals]
            for c in combos:
                kw = dict(c)
                calls.append((f"{mod.__name__}::{name}{kw}", (lambda f=f, kw=kw: f(**kw))))
    return calls


def _failing_pins():
    failed = []
    for name, call in _pin_calls():
        try:
            with warnings.catch_warnings(), np.errstate(all="ignore"):
                warnings.simplefilter("ignore")
                call()
        except Exception:                     # an assertion, or the mutant crashing a pin
            failed.append(name)
    return failed


def test_pins_pass_on_the_unmodified_oracle():
    assert _failing_pins() == []


@pytest.mark.parametrize("case,module,func,edits", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_planted_mistake_fails_a_pin(case, module, func, edits):
    with _planted(module, func, edits):
        caught = _failing_pins()
    assert caught, f"no pin notices the planted mistake {case!r} in oracle.{module}.{func}"


def test_every_mutated_function_is_restored():
    before = {(m.__name__, k): v for m in _oracle_modules() for k, v in vars(m).items()}
    for case, module, func, edits in MUTANTS[:3]:
        with _planted(module, func, edits):
            pass
    after = {(m.__name__, k): v for m in _oracle_modules() for k, v in vars(m).items()}
    assert all(after[key] is val for key, val in before.items())


def test_mutant_ids_are_unique():
    ids = [m[0] for m in MUTANTS]
    assert len(ids) == len(set(ids))
    assert not [k for k, g in itertools.groupby(sorted(ids)) if len(list(g)) > 1]
