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
    "values read from the key pool": ("o[d] += p * kv_value(jb, jb->v_pool, jb->v_scale, block, g, slot, d);",
                                      "o[d] += p * kv_value(jb, jb->k_pool, jb->k_scale, block, g, slot, d);"),
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
    "int8 codes read unsigned": ("if (jb->kv_dtype == KV_INT8) return (double)((const int8_t*)pool)[i] * (double)scl[si];",
                                 "if (jb->kv_dtype == KV_INT8) return (double)((const uint8_t*)pool)[i] * (double)scl[si];"),
    "swap-out shares no host block": ("      } else if (out) {\n        a->host_refcount[map[b]] += 1;",
                                      "      } else if (0) {\n        a->host_refcount[map[b]] += 1;"),
    "swap-in keeps the host blocks": ("        else\n          drop_host_block(a, from[lb]);", "        else\n          (void)0;"),
    "token slot shifted": ("    slot = j % ORACLE_BLOCK;\n    if (block < 0 || block >= jb->num_blocks) {",
                           "    slot = (j + 1) % ORACLE_BLOCK;\n    if (block < 0 || block >= jb->num_blocks) {"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation site not unique: {name}"
    mutant_c = tmp_path / "mutant.c"
    mutant_c.write_text(src.replace(old, new))
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off", "-pthread",
                    str(mutant_c), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle_pins.py"), "-x", "-q",
                        "-p", "no:cacheprovider"], cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, f"the pins did not catch: {name}\n{r.stdout[-2000:]}"
