"""The oracle's pins must catch plausible mistakes.

Each case plants one mistake in a copy of the oracle's C source (on the CPU,
in a temporary directory), builds it, and runs the pin suite against that
build; the suite must fail. The committed oracle itself is never modified.
"""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRCS = {"smoe": os.path.join(ROOT, "oracle", "smoe_oracle.c"), "gdn": os.path.join(ROOT, "oracle", "gdn_oracle.c")}
PINS = [os.path.join(ROOT, "tests", "test_oracle_pins.py"), os.path.join(ROOT, "tests", "test_oracle_gdn.py")]

MUTATIONS = {
    "gate_up_swapped": ("hbuf[i] = silu(g) * u;", "hbuf[i] = silu(u) * g;"),
    "down_transposed": ("acc += D[(size_t)o * I + i] * hbuf[i];",
                        "acc += D[(size_t)i * H + o] * hbuf[i];"),
    "shared_term_dropped": ("o[c] += gate[t] * y[c];", "o[c] += 0.0 * gate[t] * y[c];"),
    "tie_to_higher_id": ("(best < 0 || p[e] > p[best])", "(best < 0 || p[e] >= p[best])"),
    "no_renormalise": ("w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]] / psum;",
                       "w[(size_t)t * k + j] = p[ids[(size_t)t * k + j]];"),
    "nibble_order_reversed": ("unsigned nib = (word >> (4 * (c % 8))) & 15u;",
                              "unsigned nib = (word >> (4 * (7 - c % 8))) & 15u;"),
    "scale_bias_swapped": ("W[(size_t)r * cols + c] = sc * (double)nib + bi;",
                           "W[(size_t)r * cols + c] = bi * (double)nib + sc;"),
    "gate_sigmoid_sign": ("gate[t] = 1.0 / (1.0 + exp(-gs));", "gate[t] = 1.0 / (1.0 + exp(gs));"),
    "silu_sign": ("return v / (1.0 + exp(-v));", "return v / (1.0 + exp(v));"),
    "logit_bias_sign": ("acc += (double)bias[e];", "acc -= (double)bias[e];"),
    "wrong_group_index": ("double sc = orc_f16_to_f64(s[(size_t)r * gpr + c / ORC_GROUP]);",
                          "double sc = orc_f16_to_f64(s[(size_t)r * gpr + (c / ORC_GROUP + 1) % gpr]);"),
    "truncating_round": ("double r = nearbyint(v / quantum) * quantum;",
                         "double r = trunc(v / quantum) * quantum;"),
    "fp16_exponent_bias": ("v = ldexp(1.0 + m / 1024.0, e - 15);", "v = ldexp(1.0 + m / 1024.0, e - 16);"),
    "byte_order_reversed_8_bit": ("unsigned byte = (word >> (8 * (c % 4))) & 255u;",
                                  "unsigned byte = (word >> (8 * (3 - c % 4))) & 255u;"),
    "dense_combine_shared_term_dropped": ("o[c] += y[c] * gate[t];", "o[c] += 0.0 * y[c] * gate[t];"),
    "router_row_col_swapped": ("acc += orc_bf16_to_f64(xt[h]) * orc_bf16_to_f64(Wr[(size_t)e * H + h]);",
                               "acc += orc_bf16_to_f64(xt[h]) * orc_bf16_to_f64(Wr[(size_t)h * E + e % E]);"),
    # the Gated DeltaNet step (gdn_oracle.c)
    "gdn_decay_missing_on_read": ("double c = bt * (orc_bf16_to_f64(vv[i]) - alpha * u);",
                                  "double c = bt * (orc_bf16_to_f64(vv[i]) - u);"),
    "gdn_output_before_update": ("row[j] = alpha * row[j] + c * kn[j];\n                        oi += row[j] * qn[j];",
                                 "oi += row[j] * qn[j];\n                        row[j] = alpha * row[j] + c * kn[j];"),
    "gdn_key_not_unit": ("normalise(k + kq, dk, 1.0, kn);", "normalise(k + kq, dk, 2.0, kn);"),
    "gdn_query_is_key": ("normalise(q + kq, dk, scale, qn);", "normalise(k + kq, dk, scale, qn);"),
    "gdn_head_grouping": ("int hk = h / (nv / nk);", "int hk = h % nk;"),
}


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_pins_catch_planted_mistake(name, tmp_path):
    old, new = MUTATIONS[name]
    which = "gdn" if name.startswith("gdn_") else "smoe"
    srcs = []
    for key, path in SRCS.items():
        src = open(path).read()
        if key == which:
            assert src.count(old) == 1, "mutation anchor not found: " + name
            src = src.replace(old, new)
        out = tmp_path / (key + ".c")
        out.write_text(src)
        srcs.append(str(out))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fPIC", "-shared",
                    "-o", str(lib)] + srcs + ["-lm"], check=True)
    env = dict(os.environ, SMOE_ORACLE_LIB=str(lib))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider"] + PINS,
                       env=env, cwd=ROOT, capture_output=True, text=True, timeout=600)
    assert r.returncode != 0, "pins did not catch mutation %s:\n%s" % (name, r.stdout[-2000:])
