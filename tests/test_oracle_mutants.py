"""Plant plausible mistakes in copies of the oracle source (CPU only) and check that
the pins in test_oracle.py reject every one of them."""
import os
import subprocess
import sys

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
SRC = os.path.join(ROOT, "oracle", "indexer_topk_oracle.c")

MUTANTS = {
    "relu_dropped": ("double relu = dot > 0.0 ? dot : 0.0;", "double relu = dot;"),
    "w_transposed": ("(double)p->w[(int64_t)t * p->H + h]", "(double)p->w[((int64_t)h * p->T + t) % ((int64_t)p->T * p->H)]"),
    "q_transposed": ("const uint16_t* qr = p->q + ((int64_t)t * p->H + h) * p->D;",
                     "const uint16_t* qr = p->q + (int64_t)t * p->H * p->D + h;"),
    "k_transposed": ("dot += bf16_to_double(qr[d]) * bf16_to_double(kr[d]);",
                     "dot += bf16_to_double(qr[d]) * bf16_to_double(p->k[((int64_t)d * p->Tkv + s) % ((int64_t)p->Tkv * p->D)]);"),
    "tie_break_reversed": ("return a->id > b->id;\n}", "return a->id < b->id;\n}"),
    "causal_off_by_one": ("*n_vis = pos + 1;", "*n_vis = pos;"),
    "default_offset_top_left": ("int32_t off = p->q_causal_offsets ? p->q_causal_offsets[b] : tk - tq;\n  int32_t pos",
                                "int32_t off = p->q_causal_offsets ? p->q_causal_offsets[b] : 0;\n  int32_t pos"),
    "fill_score_zero": ("scores[r] = -INFINITY;", "scores[r] = 0.0f;"),
    "fill_id_zero": ("ids[r] = -1;", "ids[r] = 0;"),
    "ascending_order": ("if (a->score != b->score) return a->score > b->score;",
                        "if (a->score != b->score) return a->score < b->score;"),
    "weight_ignored": ("acc += (double)p->w[(int64_t)t * p->H + h] * relu;", "acc += relu;"),
    "topk_clamp_wrong": ("int32_t keff = nv < p->top_k ? nv : p->top_k;\n      int32_t* oi",
                         "int32_t keff = p->top_k > nv ? nv - 1 : p->top_k;\n      int32_t* oi"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_reject_mutant(name, tmp_path, oracle_mod):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) >= 1, f"mutation site for {name} not found"
    mutated = src.replace(old, new)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "mutant.so"
    subprocess.run(["gcc", *oracle_mod.CFLAGS, str(c), "-o", str(so), "-lm"], check=True)
    env = dict(os.environ, DTK_ORACLE_LIB=str(so))
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        os.path.join(HERE, "test_oracle.py")], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode != 0, f"mutant {name} survived the pins:\n{r.stdout[-2000:]}"
