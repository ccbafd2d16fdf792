"""The pins must catch plausible mistakes in the oracle.  Each case plants one
mistake in a copy of the oracle's C source (on the CPU, in a temporary
directory), builds it, and runs the pin suite against it: the suite must fail."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "pkv_oracle.c")

MUTANTS = {
    "e4m3 ties away from zero": ("if (rem > 0.5 || (rem == 0.5 && (n & 1))) n++;", "if (rem >= 0.5) n++;"),
    "e4m3 subnormal exponent": ("mag = ldexp((double)m, -9);", "mag = ldexp((double)m, -8);"),
    "quantiser divides by 240": ("s = (amax == 0.0f) ? 1.0f : amax / 448.0f;", "s = (amax == 0.0f) ? 1.0f : amax / 240.0f;"),
    "sliding window off by one": ("return dist <= window;", "return dist < window;"),
    "streaming window off by one": ("return j < num_sinks || j >= L - window;", "return j < num_sinks || j > L - window;"),
    "GQA maps head modulo kv heads": ("int G = jb->H / jb->Hk, g = h / G,", "int G = jb->H / jb->Hk, g = h % jb->Hk,"),
    "softmax not normalised": ("p = exp(s[j] - lse);", "p = exp(s[j] - m);"),
    "values read from the key pool": ("o[d] += p * kv_value(jb, jb->v_pool, jb->v_scale, jb->v_channel, block, g, slot, d);",
                                      "o[d] += p * kv_value(jb, jb->k_pool, jb->k_scale, jb->k_channel, block, g, slot, d);"),
    "lse off by a constant": ("lse = m + log(sum);", "lse = m + log(sum) + 1e-6;"),
    "H2O sum instead of mean over heads": ("acc[(size_t)b * acc_stride + j] += cur / (double)H;",
                                           "acc[(size_t)b * acc_stride + j] += cur;"),
    "H2O ties to the higher position": ("return (x->pos > y->pos) - (x->pos < y->pos);",
                                        "return (x->pos < y->pos) - (x->pos > y->pos);"),
    "copy-on-write never fires": ("} else if (w->refcount[row[lb]] > 1) {", "} else if (w->refcount[row[lb]] > 2) {"),
    "fork does not take references": ("if (b >= 0) a->refcount[b] += 1;", "if (b >= 0) a->refcount[b] += 0;"),
    "splitmix64 increment": ("uint64_t z = (*state += 0x9E3779B97F4A7C15ULL);", "uint64_t z = (*state += 0x9E3779B97F4A7C17ULL);"),
    "combined rule: window one short": ("const int is_sink = j < sinks, is_recent = j >= L - window;",
                                        "const int is_sink = j < sinks, is_recent = j > L - window;"),
    "combined rule: one heavy hitter short": ("for (j = 0; j < heavy && j < L; j++) heavy_hit[c[j].pos] = 1;",
                                              "for (j = 0; j + 1 < heavy && j < L; j++) heavy_hit[c[j].pos] = 1;"),
    "compaction keeps the old blocks": ("      if (*e >= 0) drop_block(w, *e);\n      *e = -1;",
                                        "      *e = -1;"),
    "int8 quantiser divides by 128": ("s = (amax == 0.0f) ? 1.0f : amax / 127.0f;",
                                      "s = (amax == 0.0f) ? 1.0f : amax / 128.0f;"),
    "int8 codes truncate": ("  n = round_half_even(a);\n  if (n > 127) n = 127;", "  n = (int)a;\n  if (n > 127) n = 127;"),
    "int8 codes read unsigned": ("if (jb->kv_dtype == KV_INT8) return (double)((const int8_t*)pool)[i] * (double)scl[si] * c;",
                                 "if (jb->kv_dtype == KV_INT8) return (double)((const uint8_t*)pool)[i] * (double)scl[si] * c;"),
    "swap-out shares no host block": ("      } else if (out) {\n        a->host_refcount[map[b]] += 1;",
                                      "      } else if (0) {\n        a->host_refcount[map[b]] += 1;"),
    "swap-in keeps the host blocks": ("        else\n          drop_host_block(a, from[lb]);", "        else\n          (void)0;"),
    "token slot shifted": ("    slot = j % ORACLE_BLOCK;\n    if (block < 0 || block >= jb->num_blocks) {",
                           "    slot = (j + 1) % ORACLE_BLOCK;\n    if (block < 0 || block >= jb->num_blocks) {"),
    "H2O select: recent window one short": ("for (j = ncand; j < L; j++) chosen[j] = 1;",
                                            "for (j = ncand + 1; j < L; j++) chosen[j] = 1;"),
    "H2O select: one heavy hitter short": ("for (j = 0; j < keep; j++) chosen[c[j].pos] = 1;",
                                           "for (j = 0; j + 1 < keep; j++) chosen[c[j].pos] = 1;"),
    "H2O update reads head 0's lse": ("- lse[(size_t)b * H + h]);", "- lse[(size_t)b * H]);"),
    "H2O update weighs masked positions": (
        "      if (!oracle_keep(L, mask_mode, num_sinks, window, j)) continue;\n      for (h = 0; h < H; h++) {",
        "      if (0) continue;\n      for (h = 0; h < H; h++) {"),
    "decode ignores the softmax scale": ("s[j] = jb->scale * dot;", "s[j] = dot;"),
    "decode averages values uniformly": ("    p = exp(s[j] - lse);\n", "    p = exp(s[j] - lse) * 0 + 1.0 / L;\n"),
    "FP8 codes read without their scale": (
        "return oracle_e4m3_decode(((const uint8_t*)pool)[i]) * (double)scl[si] * c;",
        "return oracle_e4m3_decode(((const uint8_t*)pool)[i]) * c;"),
    "channel quantiser multiplies by the channel scale": (
        "    y = c ? bf16_bits_to_float(x[d]) / c[d] : bf16_bits_to_float(x[d]);",
        "    y = c ? bf16_bits_to_float(x[d]) * c[d] : bf16_bits_to_float(x[d]);"),
    "channel quantiser's absmax ignores the channel scales": (
        "    const float v = c ? bf16_bits_to_float(x[d]) / c[d] : bf16_bits_to_float(x[d]);",
        "    const float v = bf16_bits_to_float(x[d]);"),
    "dequantisation ignores the channel scale": (
        "    double c = channel ? (double)channel[(size_t)g * jb->D + d] : 1.0;", "    double c = 1.0;"),
    "dequantisation takes kv head 0's channel scales": (
        "    double c = channel ? (double)channel[(size_t)g * jb->D + d] : 1.0;",
        "    double c = channel ? (double)channel[d] : 1.0;"),
    "quantiser takes kv head 0's channel scales": (
        "oracle_quantize_row_channel(row, q->D, q->channel + (size_t)g * q->D, q->kv_dtype, q->pool + di,",
        "oracle_quantize_row_channel(row, q->D, q->channel, q->kv_dtype, q->pool + di,"),
    "bf16 query loses its low mantissa bits": ("  return bf16_bits_to_double(((const uint16_t*)jb->q)[i]);",
                                               "  return bf16_bits_to_double(((const uint16_t*)jb->q)[i] & 0xFF00);"),
    "e4m3 saturates at 240": ("if (a >= 448.0) return (uint8_t)(sign | 0x7E);", "if (a >= 240.0) return (uint8_t)(sign | 0x77);"),
    "pool layout: slot outside kv head": ("return (((size_t)block * Hk + g) * ORACLE_BLOCK + slot) * D + d;",
                                          "return (((size_t)block * ORACLE_BLOCK + slot) * Hk + g) * D + d;"),
    "truncate frees one block too few": ("  for (lb = keep_blk; lb < nblk; lb++) {", "  for (lb = keep_blk + 1; lb < nblk; lb++) {"),
    "eviction ignores a block's last token": ("for (j = lo; j < hi && j < L; j++)", "for (j = lo; j + 1 < hi && j < L; j++)"),
    "combined rule: one sink short": ("const int is_sink = j < sinks,", "const int is_sink = j + 1 < sinks,"),
    "sequence id: largest free": ("  for (s = 0; s < a->max_seqs; s++) {\n    if (!a->active[s]) {",
                                  "  for (s = a->max_seqs - 1; s >= 0; s--) {\n    if (!a->active[s]) {"),
    "freed block goes to the back of the pool": (
        "  if (a->refcount[b] == 0) a->free_stack[a->free_top++] = b;",
        "  if (a->refcount[b] == 0) {\n    memmove(a->free_stack + 1, a->free_stack, sizeof(int32_t) * a->free_top);\n"
        "    a->free_stack[0] = b;\n    a->free_top++;\n  }"),
    "swap copies in the wrong direction": ("        pairs_out[2 * npairs] = b;\n        pairs_out[2 * npairs + 1] = map[b];",
                                           "        pairs_out[2 * npairs] = map[b];\n        pairs_out[2 * npairs + 1] = b;"),
    "compaction takes no fresh blocks": (
        "    for (k = 0; k < nb; k++) new_blocks[pos++] = take_block(w);\n  }\n  for (i = 0; i < n; i++) {",
        "    for (k = 0; k < nb; k++) new_blocks[pos++] = 0;\n  }\n  for (i = 0; i < n; i++) {"),
    "FP8 quantiser's absmax ignores the sign": (
        "    float v = fabsf(bf16_bits_to_float(x[d]));\n    if (v > amax) amax = v;\n  }\n"
        "  s = (amax == 0.0f) ? 1.0f : amax / 448.0f;",
        "    float v = bf16_bits_to_float(x[d]);\n    if (v > amax) amax = v;\n  }\n"
        "  s = (amax == 0.0f) ? 1.0f : amax / 448.0f;"),
    "INT8 quantiser's absmax ignores the sign": (
        "    float v = fabsf(bf16_bits_to_float(x[d]));\n    if (v > amax) amax = v;\n  }\n"
        "  s = (amax == 0.0f) ? 1.0f : amax / 127.0f;",
        "    float v = bf16_bits_to_float(x[d]);\n    if (v > amax) amax = v;\n  }\n"
        "  s = (amax == 0.0f) ? 1.0f : amax / 127.0f;"),
    "INT8 codes lose their sign": ("return (int8_t)(x < 0.0f ? -n : n);", "return (int8_t)n;"),
    "quantised scale stored at the neighbouring slot": (
        "      size_t si = ((size_t)block * q->Hk + g) * ORACLE_BLOCK + slot;",
        "      size_t si = ((size_t)block * q->Hk + g) * ORACLE_BLOCK + (slot ^ 1);"),
    "scatter reverses the kv heads": ("      size_t s = (((size_t)t * Hk + g) * D) * (size_t)elem_bytes;",
                                      "      size_t s = (((size_t)t * Hk + (Hk - 1 - g)) * D) * (size_t)elem_bytes;"),
    "row copy leaves the K scale": (
        "        k_scale[((size_t)db * Hk + g) * ORACLE_BLOCK + dso] = k_scale[((size_t)sb * Hk + g) * ORACLE_BLOCK + so];",
        "        (void)0;"),
    "block copy leaves V": (
        "  memcpy((char*)v_pool + (size_t)dst * blk, (char*)v_pool + (size_t)src * blk, blk);\n"
        "  if (k_scale && v_scale) {\n    size_t sb",
        "  if (k_scale && v_scale) {\n    size_t sb"),
    "block copy leaves the K scales": (
        "    memcpy(k_scale + (size_t)dst * sb, k_scale + (size_t)src * sb, sb * sizeof(float));", "    (void)0;"),
    "swap copy leaves the V scales": ("      memcpy(dst_vs + d * sb, src_vs + s * sb, sb * sizeof(float));", "      (void)0;"),
    "e4m3 decode with exponent bias 8": ("    mag = ldexp((double)(8 + m), e - 10); /* (1 + m/8) * 2^(e-7) */",
                                         "    mag = ldexp((double)(8 + m), e - 11);"),
    "e4m3 encode loses negative zero": ("  sign = signbit(x) ? 0x80 : 0x00;", "  sign = (x < 0) ? 0x80 : 0x00;"),
    "swap-in shares no device block": ("      } else {\n        a->refcount[map[b]] += 1;\n      }",
                                       "      } else {\n        (void)0;\n      }"),
    "swap never marks sequences": ("    a->swapped[s] = out ? 1 : 0;", "    a->swapped[s] = 0;"),
    "fork shares full blocks only": (
        "  nblk = (a->lens[src] + ORACLE_BLOCK - 1) / ORACLE_BLOCK;\n  for (lb = 0; lb < nblk; lb++) {\n"
        "    int b = a->tables[(size_t)src",
        "  nblk = a->lens[src] / ORACLE_BLOCK;\n  for (lb = 0; lb < nblk; lb++) {\n    int b = a->tables[(size_t)src"),
    "softmax sum without the running max": (
        "    if (oracle_keep(L, jb->mask_mode, jb->num_sinks, jb->window, j)) sum += exp(s[j] - m);",
        "    if (oracle_keep(L, jb->mask_mode, jb->num_sinks, jb->window, j)) sum += exp(s[j]);"),
    "combined rule ranks only positions before the window": (
        "  qsort(c, (size_t)L, sizeof(scored_pos), cmp_desc_score_asc_pos);",
        "  qsort(c, (size_t)(L > window ? L - window : 0), sizeof(scored_pos), cmp_desc_score_asc_pos);"),
}


def _run_mutant(name, work):
    """Builds the oracle with one planted mistake and runs the pins against
    it; returns (pins failed?, the end of their output)."""
    old, new = MUTANTS[name]
    src = open(SRC).read()
    if src.count(old) != 1:
        return None, f"mutation site not unique: {name}"
    d = work / f"m{sorted(MUTANTS).index(name)}"
    d.mkdir()
    mutant_c, so = d / "mutant.c", d / "libmutant.so"
    mutant_c.write_text(src.replace(old, new))
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off", "-pthread",
                    str(mutant_c), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(so), OMP_NUM_THREADS="1")
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    return r.returncode != 0, r.stdout[-2000:]


@pytest.fixture(scope="module")
def mutant_results(tmp_path_factory):
    """Every mutant's pin run, several at a time (each is an independent
    process on its own copy of the oracle)."""
    from concurrent.futures import ThreadPoolExecutor
    work = tmp_path_factory.mktemp("mutants")
    names = sorted(MUTANTS)
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as ex:
        return dict(zip(names, ex.map(lambda n: _run_mutant(n, work), names)))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, mutant_results):
    caught, tail = mutant_results[name]
    assert caught is not None, tail
    assert caught, f"the pins did not catch: {name}\n{tail}"
