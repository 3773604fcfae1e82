"""Plant plausible mistakes in copies of the oracle source; each must fail a pin.

Every mutant is one textual edit of `oracle/tts_oracle.c` (a dropped term, a
wrong sign, index or operand, an off-by-one).  The copy is compiled into a
temporary library and all pins of `oracle_pins` run against it in a child
process; the test passes when at least one pin fails.  The real oracle is
never modified.
"""
import json
import os
import subprocess
import sys
import tempfile
from concurrent.futures import ThreadPoolExecutor
from pathlib import Path

import pytest

import oracle

ROOT = Path(__file__).resolve().parents[1]

MUTANTS = [
    ("philox: low product word in place of the high one", "uint64_t y1 = lo1;", "uint64_t y1 = hi1;"),
    ("philox: second key word not bumped", "        k1 += W1;\n", ""),
    ("philox: nine rounds", "round < 10", "round < 9"),
    ("philox: words 1 and 3 swapped in the xor", "uint64_t y0 = hi1 ^ x1 ^ k0;", "uint64_t y0 = hi1 ^ x3 ^ k0;"),
    ("uniform: wrong bit window", "const uint32_t k = half >> 9;", "const uint32_t k = half >> 10;"),
    ("uniform: high half first",
     "(lane & 1u) ? (uint32_t)(word >> 32) : (uint32_t)word", "(lane & 1u) ? (uint32_t)word : (uint32_t)(word >> 32)"),
    ("uniform: counter block index", "const uint64_t ctr[4] = {idx / 8u, tag, pos, 0};",
     "const uint64_t ctr[4] = {idx / 4u, tag, pos, 0};"),
    ("gumbel: sign", "return -logf(-logf(u));", "return logf(-logf(u));"),
    ("append: slot offset", "+ s % ORC_BLOCK) * row;", "+ (s + 1) % ORC_BLOCK) * row;"),
    ("append: logical block", "s / ORC_BLOCK];\n            if (blk < 0 || blk >= num_blocks) return -1;",
     "(s + 1) / ORC_BLOCK];\n            if (blk < 0 || blk >= num_blocks) return -1;"),
    ("fp8 append: logical block", "const int logical = s / ORC_BLOCK;", "const int logical = (s + 1) / ORC_BLOCK;"),
    ("attn: scale dropped", "s[t] = scale * dot;", "s[t] = dot;"),
    ("attn: GQA head mapping", "const int g = h / group;", "const int g = h % Hkv;"),
    ("attn: causal limit off by one", "causal ? L - q_len + j + 1 : L", "causal ? L - q_len + j + 2 : L"),
    ("attn: causal limit short", "causal ? L - q_len + j + 1 : L", "causal ? L - q_len + j : L + 0"),
    ("attn: key slot", "kv(ctx, 0, blk, g, t % ORC_BLOCK, d)", "kv(ctx, 0, blk, g, (t + 1) % ORC_BLOCK, d)"),
    ("attn: values from the key pool", "o[d] += p * kv(ctx, 1,", "o[d] += p * kv(ctx, 0,"),
    ("attn: unnormalised weights", "const double p = s[t] / denom;", "const double p = s[t];"),
    ("head: W transposed", "load_elem(W, (size_t)v * H + k, is_bf16)", "load_elem(W, (size_t)k * V + v, is_bf16)"),
    ("head: highest index wins ties", "if (arg < 0 || key > top) {", "if (arg < 0 || key >= top) {"),
    ("head: eos mask ignored", "mask[r] = eos_allowed[r] ? 1u : 0u;", "mask[r] = 1u;"),
    ("head: temperature multiplies", "key = logit / T + orc_gumbel", "key = logit * T + orc_gumbel"),
    ("head: noise indexed by row", "orc_gumbel(seed[r], step[r], 0u, pos, (uint32_t)v)",
     "orc_gumbel(seed[r], step[r], 0u, pos, (uint32_t)r)"),
    ("head: counter position ignored", "return head_select_at(h, W, is_bf16, b, R, H, V, mode, T, seed, step, 0u,",
     "return head_select_at(h, W, is_bf16, b, R, H, V, mode, T, seed, step, 1u,"),
    ("predictor: attention one token short", "for (int t = 0; t <= i; ++t) {\n                    double dot",
     "for (int t = 0; t < i || t == 0; ++t) {\n                    double dot"),
    ("predictor: embedding of the next codebook", "const uint16_t *Ei = E + (size_t)i * V * H;",
     "const uint16_t *Ei = E + (size_t)(i + 1 < n_steps ? i + 1 : i) * V * H;"),
    ("predictor: Gumbel position of the step", "(uint32_t)(i + 1), 0, NULL", "(uint32_t)i, 0, NULL"),
    ("predictor: projection not rounded", "qkv[f] = load_elem(&b, 0, 1);", "qkv[f] = acc + 0.0 * b;"),
    ("predictor: values read from the keys", "acc += sc[t] / denom * vc[", "acc += sc[t] / denom * kc["),
    ("predictor: GQA map", "const int kvh = h / group;", "const int kvh = h % Hkv;"),
    ("verify: accept test reversed", "accepted = u < ratio;", "accepted = u > ratio;"),
    ("verify: zero draft probability accepted", "if (dp[d] > 0.0f) {", "if (dp[d] >= 0.0f) {"),
    ("verify: residual not clamped", "fmaxf(pt[v] - dp[v], 0.0f)", "fabsf(pt[v] - dp[v])"),
    ("verify: residual ignores the draft", "fmaxf(pt[v] - dp[v], 0.0f)", "pt[v]"),
    ("verify: does not stop at the first rejection", "rejected = 1;\n            break;", "rejected = 1;"),
    ("verify: temperature dropped", "row_probs(tl, V, T, pt);", "row_probs(tl, V, 1.0f, pt);"),
    ("rope: rotation sign", "out[(size_t)r * D + i] = (float)(x1 * c - x2 * sn);",
     "out[(size_t)r * D + i] = (float)(x1 * c + x2 * sn);"),
    ("rope: frequency exponent", "pow(base, -2.0 * i / D)", "pow(base, -1.0 * i / D)"),
    ("rope: pairs of neighbours", "const double x2 = load_elem(x, (size_t)r * D + i + h, is_bf16);",
     "const double x2 = load_elem(x, (size_t)r * D + (i ^ 1), is_bf16);"),
    ("rope: position off by one", "const double a = (double)pos[r] * pow", "const double a = (double)(pos[r] + 1) * pow"),
    ("e4m3: ties to the later code", "(err == best_err && (c & 1) == 0)", "(err == best_err)"),
    ("e4m3: largest finite code excluded", "for (int c = 0; c <= 0x7E; ++c)", "for (int c = 0; c < 0x7E; ++c)"),
    ("e4m3: subnormal exponent", "ldexp((double)m, -9)", "ldexp((double)m, -10)"),
    ("fp8 append: scale for a maximum of 240", "amax / 448.0f", "amax / 240.0f"),
    ("fp8 append: value slots in natural order", "return (size_t)(2048 + 16 * d + v_pos(s));",
     "return (size_t)(2048 + 16 * d + s);"),
    ("fp8 append: keys unswizzled", "16 * ((d / 16) ^ (s % 8))", "16 * (d / 16)"),
    ("fp8 attn: values scaled by the key scale", "memcpy(&sc, tile + (is_v ? 4160 : 4096) + 4 * slot, 4);",
     "memcpy(&sc, tile + 4096 + 4 * slot, 4);"),
    ("mish: softplus without the logarithm", "log1p(exp(x))", "exp(x)"),
    ("mish: sign inside tanh", "return x * tanh(sp);", "return x * tanh(-sp);"),
    ("bf16 rounding: truncation", "nearbyint(ldexp(m, 8))", "trunc(ldexp(m, 8))"),
    ("bf16 rounding: one bit too many", "nearbyint(ldexp(m, 8))", "nearbyint(ldexp(m, 9))"),
    ("audio expand: bias dropped", "double acc = b1 ? (double)b1[f] : 0.0;", "double acc = 0.0;"),
    ("audio expand: W1 transposed", "load_elem(W1, (size_t)f * H + k, 1)", "load_elem(W1, (size_t)k * F + f, 1)"),
    ("masked head: bias dropped", "double acc = b ? (double)b[v] : 0.0;", "double acc = 0.0;"),
    ("masked head: tail offset", "const int j = v - (V - n_tail);", "const int j = v - (V - n_tail) - 1;"),
    ("masked head: mask bits reversed", "!((tail_allowed[r] >> j) & 1u)",
     "!((tail_allowed[r] >> (n_tail - 1 - j)) & 1u)"),
    ("verify: bonus always drawn", "if (!rejected && (flags & 1)) {", "if (!rejected) {"),
    ("verify: draw noise keyed by the rejected row",
     "logf(r) + orc_gumbel(seed[b], step[b], 2u, 0u, (uint32_t)v)",
     "logf(r) + orc_gumbel(seed[b], step[b], 2u, (uint32_t)i, (uint32_t)v)"),
    ("verify: bonus noise keyed by the bonus row",
     "tl[v] / T + orc_gumbel(seed[b], step[b], 2u, 0u, (uint32_t)v)",
     "tl[v] / T + orc_gumbel(seed[b], step[b], 2u, (uint32_t)K, (uint32_t)v)"),
    ("verify: bonus from the last draft row",
     "target_logits + ((size_t)b * (K + 1) + K) * V;", "target_logits + ((size_t)b * (K + 1) + K - 1) * V;"),
]

_CHILD = r"""
import json, sys
sys.path[:0] = [{root!r}, {tests!r}]
import oracle, oracle_pins
o = oracle.Oracle({lib!r})
failed = []
for check in oracle_pins.ALL_CHECKS:
    try:
        check(o)
    except Exception as e:  # a failed pin
        failed.append(check.__name__)
print(json.dumps(failed))
"""


def _run_mutant(tmp: Path, i: int, old: str, new: str):
    src = oracle.SRC.read_text()
    assert src.count(old) == 1, f"mutant {i}: snippet must occur exactly once: {old!r}"
    msrc = tmp / f"mutant_{i}.c"
    msrc.write_text(src.replace(old, new))
    lib = oracle.build(msrc, tmp / f"libmutant_{i}.so", force=True)
    code = _CHILD.format(root=str(ROOT), tests=str(ROOT / "tests"), lib=str(lib))
    env = dict(os.environ, OMP_NUM_THREADS="1")
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True,
                       timeout=600, env=env)
    if p.returncode != 0:
        return ["<child crashed: " + p.stderr.strip().splitlines()[-1][:200] + ">"]
    return json.loads(p.stdout.strip().splitlines()[-1])


def test_every_mutant_fails_a_pin():
    with tempfile.TemporaryDirectory() as d:
        tmp = Path(d)
        with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 2)) as ex:
            futs = [ex.submit(_run_mutant, tmp, i, old, new) for i, (_, old, new) in enumerate(MUTANTS)]
            results = [f.result() for f in futs]
    survivors = [MUTANTS[i][0] for i, failed in enumerate(results) if not failed]
    assert not survivors, f"mistakes no pin catches: {survivors}"


@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_snippet_present(name, old, new):
    assert oracle.SRC.read_text().count(old) == 1
