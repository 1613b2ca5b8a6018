"""The oracle's pins must be able to fail.

Each case below plants one plausible mistake in a copy of oracle/ep_oracle.c
(a dropped term, a wrong rounding constant, a reversed order, a wrong index,
a flipped sign, a misread of the pages), compiles the copy with gcc, runs every
pin of test_oracle_pins.py and test_oracle_dtypes.py against it, and requires
that at least one pin fails.  The unmodified source must pass the same run, so
a harness fault cannot pass for a caught mistake.

A change that is not a mistake is left out: "x > 0x477FF000" in place of
">=" in the binary16 overflow test, for instance, gives the same result,
because 65520 (the tie between 65504 and 2^16) carries into infinity through
the ordinary rounding path too.

Every planted mistake keeps all memory accesses inside the buffers the Python
wrappers allocate (no mutant reads or writes past an array), so a mutant fails
by a wrong value, never by a crash.  CPU only.
"""
from __future__ import annotations

import concurrent.futures
import inspect
import itertools
import os
import subprocess

import pytest
from _pytest.mark.structures import ParameterSet

import oracle
import test_oracle_dtypes
import test_oracle_pins
import test_oracle_rm_pins
import test_oracle_shard_pins

SRC = os.path.join(os.path.dirname(os.path.abspath(oracle.__file__)), "ep_oracle.c")

# (name, original text, planted text, which occurrence of the original)
MUTANTS = [
    # binary32 -> bfloat16
    ("bf16_round_half_up", "u += 0x7FFFu + lsb;", "u += 0x8000u + 0u * lsb;", 0),
    ("bf16_truncate", "u += 0x7FFFu + lsb;", "u += 0u * lsb;", 0),
    ("bf16_nan_not_quieted", "return (uint16_t)((u >> 16) | 0x0040u);", "return (uint16_t)(u >> 16);", 0),
    # binary16 <-> binary32
    ("f16_round_half_up", "uint32_t r = x + 0x0FFFu + ((x >> 13) & 1u);", "uint32_t r = x + 0x1000u;", 0),
    ("f16_subnormal_ties_away", "if (rem > half || (rem == half && (q & 1u))) q += 1u;",
     "if (rem >= half) q += 1u;", 0),
    ("f16_overflow_from_max", "if (x >= 0x477FF000u)", "if (x >= 0x477FE000u)", 0),
    ("f16_no_overflow_check", "if (x >= 0x477FF000u) return", "if (x >= 0xFFFFFFFFu) return", 0),
    ("f16_widen_subnormal_exponent", "127 - 15 + 1 - shift", "127 - 15 - shift", 0),
    ("f16_payload_loaded_as_bf16", "if (dtype == 1) return oracle_f16_to_f32(",
     "if (dtype == 1) return oracle_bf16_to_f32(", 0),
    ("f16_payload_rounded_as_bf16", "else if (dtype == 1) ((uint16_t*)base)[i] = oracle_f32_to_f16(v);",
     "else if (dtype == 1) ((uint16_t*)base)[i] = oracle_f32_to_bf16(v);", 0),
    # prepare
    ("prepare_no_padding", "int64_t padded = ((c + A - 1) / A) * A;", "int64_t padded = c;", 0),
    ("prepare_last_in_first_out", "int64_t s = cursor[e]++;",
     "int64_t s = offsets[e] + token_counts[e] - 1 - (cursor[e]++ - offsets[e]);", 0),
    ("prepare_overflow_at_equal", "if (P > R) status", "if (P >= R) status", 0),
    ("prepare_bad_index_not_flagged", "{ status |= STATUS_BAD_INDEX; continue; }", "{ continue; }", 0),
    ("prepare_masked_flagged_bad", "if (e == -1) continue;",
     "if (e == -1) { status |= STATUS_BAD_INDEX; continue; }", 0),
    # dispatch
    ("dispatch_weight_of_first_k", "recv_topk_weights[s] = topk_weights[r];",
     "recv_topk_weights[s] = topk_weights[r - r % K];", 0),
    ("dispatch_padding_weight_one", "recv_topk_weights[s] = 0.0f;", "recv_topk_weights[s] = 1.0f;", 0),
    ("dispatch_padding_row_not_zero", "dst[s * rb + b] = 0;", "dst[s * rb + b] = 0x3F;", 0),
    ("dispatch_bytes_swapped", "dst[s * rb + b] = src[t * rb + b];",
     "dst[s * rb + b] = src[t * rb + (b ^ 1)];", 0),
    # combine (and the token half of dispatch_bwd)
    ("combine_negative_zero_start", "float acc = 0.0f;", "float acc = -0.0f;", 0),
    ("combine_k_descending", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = K - 1; k >= 0; --k) {", 0),
    ("combine_double_accumulator", "float acc = 0.0f;", "double acc = 0.0;", 0),
    ("combine_drops_last_k", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = 0; k < K - 1; ++k) {", 0),
    # combine_bwd
    ("combine_bwd_padding_not_zero", "(r < 0) ? (unsigned char)0 :", "(r < 0) ? (unsigned char)1 :", 0),
    ("combine_bwd_bytes_swapped", "src[(int64_t)(r / K) * rb + b]", "src[(int64_t)(r / K) * rb + (b ^ 1)]", 0),
    # weight half of dispatch_bwd
    ("weight_grad_masked_negative_zero", "g_recv_topk_weights == 0) ? 0.0f :",
     "g_recv_topk_weights == 0) ? -0.0f :", 0),
    # weighted combine and its backward
    ("weighted_fused_multiply_add", "acc = acc + prod;",
     "acc = (float)((double)acc + (double)w[s] * (double)load_elem(rows, (int64_t)s * H + h, dtype));", 0),
    ("weighted_ignores_weight", "float prod = w[s] * load_elem(", "float prod = 1.0f * load_elem(", 0),
    ("weighted_k_descending", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = K - 1; k >= 0; --k) {", 1),
    ("weighted_bwd_drops_weight", "float prod = w[s] * g;", "float prod = g;", 0),
    ("weighted_bwd_weight_grad_sign", "g_w[s] = dot;", "g_w[s] = -dot;", 0),
    ("weighted_bwd_dot_of_scaled_grad", "dot += (double)g * (double)load_elem(rows",
     "dot += (double)prod * (double)load_elem(rows", 0),
    # sharded prepare and row operations
    ("shard_owner_round_robin", "int64_t q = e / Eloc;", "int64_t q = e % N;", 0),
    ("shard_no_padding", "run += ((counts[e] + A - 1) / A) * A;", "run += counts[e];", 0),
    ("shard_blocks_not_restarted_per_owner",
     "    for (int64_t q = 0; q < N; ++q) {\n        int64_t run = 0;\n",
     "    int64_t run = 0;\n    for (int64_t q = 0; q < N; ++q) {\n", 0),
    ("shard_overflow_first_rank_only",
     "for (int64_t q = 0; q < N; ++q) if (overflow) status[q] |= STATUS_OVERFLOW;",
     "if (overflow) status[0] |= STATUS_OVERFLOW;", 0),
    ("shard_overflow_at_equal", "if (run > R) overflow = 1;", "if (run >= R) overflow = 1;", 0),
    ("shard_bad_index_on_rank0", "status[rank] |= STATUS_BAD_INDEX", "status[0] |= STATUS_BAD_INDEX", 0),
    ("shard_gather_k_descending", "for (int64_t k = 0; k < K; ++k) {", "for (int64_t k = K - 1; k >= 0; --k) {", 2),
    # rank-major prepare, dispatch and weight gradients
    ("rm_owner_round_robin", "goes[e / Eloc] = 1;", "goes[e % N] = 1;", 0),
    ("rm_no_dedup", "first[i] = row_of[q] < 0;\n            if (row_of[q] < 0) {",
     "first[i] = 1;\n            if (1) {", 0),
    ("rm_overflow_at_equal", "if (M[q] > R) overflow = 1;", "if (M[q] >= R) overflow = 1;", 0),
    ("rm_bad_index_on_rank0", "if (e < -1 || e >= E) status[rank] |= STATUS_BAD_INDEX;",
     "if (e < -1 || e >= E) status[0] |= STATUS_BAD_INDEX;", 0),
    ("rm_ids_not_relative", "recv_idx[s * K + k] = mine ? e - q * Eloc : -1;",
     "recv_idx[s * K + k] = mine ? e : -1;", 0),
    ("rm_foreign_ids_kept", "recv_idx[s * K + k] = mine ? e - q * Eloc : -1;",
     "recv_idx[s * K + k] = e >= 0 && e < E ? e - q * Eloc : -1;", 0),
    ("rm_foreign_weights_kept", "recv_weights[s * K + k] = mine && topk_weights ?",
     "recv_weights[s * K + k] = topk_weights ?", 0),
    ("rm_weight_grad_first_entry", "g_of_rank[dest[i]][(int64_t)row[i] * K + k];",
     "g_of_rank[dest[i]][(int64_t)row[i] * K];", 0),
    ("shard_weight_grad_negative_zero", "(s < 0 || g_of_rank == 0) ? 0.0f :",
     "(s < 0 || g_of_rank == 0) ? -0.0f :", 0),
]


def _plant(src: str, old: str, new: str, nth: int) -> str:
    pos = -1
    for _ in range(nth + 1):
        pos = src.index(old, pos + 1)
    return src[:pos] + new + src[pos + len(old):]


def _compile(src_text: str, out_dir: str, name: str) -> str:
    c = os.path.join(out_dir, name + ".c")
    so = os.path.join(out_dir, name + ".so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-std=c99", "-O1", "-fPIC", "-shared", "-ffp-contract=off",
                    "-fno-fast-math", "-w", "-o", so, c], check=True)
    return so


def _pin_calls():
    """Every (label, function, kwargs) of the two pin modules, expanded over
    their parametrize marks."""
    calls = []
    for mod in (test_oracle_pins, test_oracle_dtypes, test_oracle_shard_pins, test_oracle_rm_pins):
        for fname, fn in sorted(vars(mod).items()):
            if not (fname.startswith("test_") and inspect.isfunction(fn)):
                continue
            axes = []
            for m in getattr(fn, "pytestmark", []):
                if m.name != "parametrize":
                    continue
                names = m.args[0]
                names = [n.strip() for n in names.split(",")] if isinstance(names, str) else list(names)
                rows = []
                for v in m.args[1]:
                    if isinstance(v, ParameterSet):
                        v = v.values
                    rows.append(dict(zip(names, v if len(names) > 1 else (v,))))
                axes.append(rows)
            params = set(inspect.signature(fn).parameters)
            for combo in itertools.product(*axes) if axes else [()]:
                kw = {}
                for part in combo:
                    kw.update(part)
                if params - set(kw) - {"oracle_mod"}:
                    continue
                if "oracle_mod" in params:
                    kw["oracle_mod"] = oracle
                calls.append(("%s.%s" % (mod.__name__, fname), fn, kw))
    return calls


def _first_failure(calls):
    for label, fn, kw in calls:
        try:
            fn(**kw)
        except Exception as e:  # a pin failed: the mistake is caught
            return "%s (%s)" % (label, type(e).__name__)
    return None


@pytest.fixture(scope="module")
def libraries(tmp_path_factory):
    base = open(SRC).read()
    for name, old, new, nth in MUTANTS:
        assert base.count(old) > nth, (name, old)
    d = str(tmp_path_factory.mktemp("oracle_mutants"))
    jobs = {"unmodified": base}
    jobs.update({name: _plant(base, old, new, nth) for name, old, new, nth in MUTANTS})
    with concurrent.futures.ThreadPoolExecutor(max_workers=8) as pool:
        futs = {n: pool.submit(_compile, text, d, n) for n, text in jobs.items()}
        return {n: f.result() for n, f in futs.items()}


@pytest.fixture(scope="module")
def pin_calls():
    calls = _pin_calls()
    assert len(calls) >= 80
    return calls


def test_unmodified_source_passes(libraries, pin_calls):
    with oracle.use_library(libraries["unmodified"]):
        assert _first_failure(pin_calls) is None


@pytest.mark.parametrize("name", [m[0] for m in MUTANTS])
def test_planted_mistake_is_caught(libraries, pin_calls, name):
    with oracle.use_library(libraries[name]):
        caught_by = _first_failure(pin_calls)
    assert caught_by is not None, "no pin fails for the planted mistake %s" % name
