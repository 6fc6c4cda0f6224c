"""Planted mistakes in copies of the oracle must each fail at least one pin.

Each mutant is a one-place edit of ``oracle/vp_oracle.c`` (a dropped term, a
flipped sign, a wrong index or operand, a missing guard) compiled into a
temporary library on the CPU. The real oracle source is never modified.
"""
import os
import shutil
import subprocess

import pytest

import oracle
from tests import pins

SRC = os.path.join(os.path.dirname(oracle.__file__), "vp_oracle.c")

MUTANTS = [
    ("entropy sign", "if (p > 0.0) H -= p * lp;", "if (p > 0.0) H += p * lp;"),
    ("entropy zero-weight guard dropped", "if (p > 0.0) H -= p * lp;", "H -= p * lp;"),
    ("log p adds log S", "return (zj - s->m) - s->logS;", "return (zj - s->m) + s->logS;"),
    ("sum-exp not centred", "s.S += exp(v - s.m);", "s.S += exp(v);"),
    ("NaN entries not flagged", "if (isnan(v) || v == INFINITY) s.bad = 1;", "if (v == INFINITY) s.bad = 1;"),
    ("logprobs ignored target not zero", "if (t < 0) { logp[r] = 0.0; continue; }",
     "if (t < 0) { logp[r] = NAN; continue; }"),
    ("vocab_start added", "int64_t loc = t - vocab_start;\n        if (loc < 0 || loc >= V) { logp[r] = NAN;",
     "int64_t loc = t + vocab_start;\n        if (loc < 0 || loc >= V) { logp[r] = NAN;"),
    ("logprobs bwd sign", "d[j] = g[r] * (onehot - p);", "d[j] = g[r] * (p - onehot);"),
    ("logprobs bwd onehot dropped", "d[j] = g[r] * (onehot - p);", "d[j] = g[r] * (0.0 - p);"),
    ("entropy bwd drops +H", "d[j] = (p > 0.0) ? -g[r] * p * (lp + H) : 0.0;",
     "d[j] = (p > 0.0) ? -g[r] * p * lp : 0.0;"),
    ("entropy bwd sign", "d[j] = (p > 0.0) ? -g[r] * p * (lp + H) : 0.0;",
     "d[j] = (p > 0.0) ? g[r] * p * (lp + H) : 0.0;"),
    ("KL wrong operand", "if (p > 0.0) kl += p * (lp - log_prob(Q[j], sq));",
     "if (p > 0.0) kl += p * (lp - log_prob(P[j], sq));"),
    ("KL direction swapped", "kl[r] = direction == 0 ? kl_row(A, B, V, &sa, &sb)",
     "kl[r] = direction == 1 ? kl_row(A, B, V, &sa, &sb)"),
    ("mismatch test swapped", "if (P[j] > -INFINITY && Q[j] == -INFINITY) return 1;",
     "if (Q[j] > -INFINITY && P[j] == -INFINITY) return 1;"),
    ("mismatch ignored", "if (mismatch(P, Q, V)) return INFINITY;", ""),
    ("KL dQ sign", "if (dQ) dQ[j] = g * (q - p);", "if (dQ) dQ[j] = g * (p - q);"),
    ("KL dP drops -KL", "else dP[j] = (p > 0.0) ? g * p * (lp - lq - kl) : 0.0;",
     "else dP[j] = (p > 0.0) ? g * p * (lp - lq) : 0.0;"),
    ("KL bwd direction swapped", "if (direction == 0) kl_bwd_row(A, B, V, g[r], dA, dB);",
     "if (direction == 1) kl_bwd_row(A, B, V, g[r], dA, dB);"),
    ("merge drops re-centring", "W += alpha * (parts[s].W - (m - parts[s].m) * parts[s].S);",
     "W += alpha * parts[s].W;"),
    ("merge zero-weight skip dropped", "if (w == 0.0) continue;                  /* zero-weight shard skipped */", ""),
    ("KL merge shift sign", "W += ap * (parts[s].W - (dp - dq) * parts[s].Sp);",
     "W += ap * (parts[s].W - (dp + dq) * parts[s].Sp);"),
    ("shard record W column", "o[0] = s.m; o[1] = s.S; o[2] = s.W; o[3] = s.bad;",
     "o[0] = s.m; o[1] = s.S; o[2] = s.S; o[3] = s.bad;"),
    ("shard KL record Q max", "o[2] = s.mq; o[3] = s.Sq;", "o[2] = s.mp; o[3] = s.Sq;"),
    ("shard KL record direction", "const double *P = (direction == 0 ? a : b) + r * V;\n        const double *Q = (direction == 0 ? b : a) + r * V;\n        shard_kl s",
     "const double *P = (direction == 1 ? a : b) + r * V;\n        const double *Q = (direction == 1 ? b : a) + r * V;\n        shard_kl s"),
    ("JSD mixture weights swapped", "double lmix = log(beta * q + (1.0 - beta) * p);\n        if (p > 0.0) kp",
     "double lmix = log((1.0 - beta) * q + beta * p);\n        if (p > 0.0) kp"),
    ("JSD teacher term dropped", "return beta * kq + (1.0 - beta) * kp;", "return (1.0 - beta) * kp;"),
    ("JSD dA drops -KL(p||mix)", "g[r] * (1.0 - beta) * p * ((lp - lmix) - ka)", "g[r] * (1.0 - beta) * p * (lp - lmix)"),
    ("JSD dB wrong weight", "g[r] * beta * q * ((lq - lmix) - kb)", "g[r] * (1.0 - beta) * q * ((lq - lmix) - kb)"),
    ("JSD endpoint directions swapped", "if (beta == 0.0) jsd[r] = kl_row(B, A, V, &sb, &sa);",
     "if (beta == 0.0) jsd[r] = kl_row(A, B, V, &sa, &sb);"),
    ("top-k duplicates overwrite", "if (t >= 0) d[t - vocab_start] += g[r * K + k];",
     "if (t >= 0) d[t - vocab_start] = g[r * K + k];"),
    ("top-k ignored ids counted", "if (t < 0) continue;\n            int64_t loc = t - vocab_start;\n            if (loc < 0 || loc >= V) bad = 1;",
     "if (t < 0) { gsum += g[r * K + k]; continue; }\n            int64_t loc = t - vocab_start;\n            if (loc < 0 || loc >= V) bad = 1;"),
    ("top-k id stride", "int64_t t = targets[r * K + k];\n            double *out", "int64_t t = targets[r + k];\n            double *out"),
    ("linear logits transposed", "acc += h[r * D + k] * W[j * D + k];", "acc += h[r * D + k] * W[k * V + j];"),
    ("linear dW wrong row", "out[k] += c * h[r * D + k];", "out[k] += c * h[((r + 1) % N) * D + k];"),
    ("linear dh wrong vocab row", "out[k] += c * W[j * D + k];", "out[k] += c * W[((j + 1) % V) * D + k];"),
    ("linear bwd onehot dropped", "z[j] = g[r] * (((j == loc) ? 1.0 : 0.0) - p);", "z[j] = g[r] * (0.0 - p);"),
    ("linear chain rule dz transposed", "double c = dz[r * V + j];", "double c = dz[j * N + r];"),
    ("linear chain rule dW from the wrong hidden column", "for (int64_t r = 0; r < N; ++r) {\n                double c = dz[r * V + j];\n                for (int64_t k = 0; k < D; ++k) out[k] += c * h[r * D + k];",
     "for (int64_t r = 0; r < N; ++r) {\n                double c = dz[r * V + j];\n                for (int64_t k = 0; k < D; ++k) out[k] += c * h[r * D + (D - 1 - k)];"),
    ("linear KL model B with model A's width", "vpo_linear_logits(hb, Wb, N, V, Db, zb);\n    vpo_kl_fwd",
     "vpo_linear_logits(hb, Wb, N, V, Da, zb);\n    vpo_kl_fwd"),
    ("linear KL bwd gradients of A and B swapped", "linear_chain_rule(ha, Wa, N, V, Da, dza, dha, dWa);",
     "linear_chain_rule(ha, Wa, N, V, Da, dzb, dha, dWa);"),
    ("linear entropy bwd reads logits as dz", "linear_chain_rule(h, W, N, V, D, dz, dh, dW);",
     "linear_chain_rule(h, W, N, V, D, logits, dh, dW);"),
    ("linear JSD models swapped", "vpo_jsd_fwd(za, zb, N, V, beta, jsd);", "vpo_jsd_fwd(zb, za, N, V, beta, jsd);"),
    ("linear JSD bwd gradients of B to A", "vpo_jsd_bwd(za, zb, N, V, beta, g, dza, dzb);\n    linear_chain_rule(ha, Wa, N, V, Da, dza, dha, dWa);",
     "vpo_jsd_bwd(za, zb, N, V, beta, g, dza, dzb);\n    linear_chain_rule(ha, Wa, N, V, Da, dzb, dha, dWa);"),
]


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


@pytest.mark.skipif(shutil.which("gcc") is None, reason="gcc not available")
@pytest.mark.parametrize("name,old,new", MUTANTS, ids=[m[0] for m in MUTANTS])
def test_mutant_is_caught(source, tmp_path, name, old, new):
    assert source.count(old) >= 1, f"mutation site not found: {old!r}"
    mutated = source.replace(old, new, 1)
    c = tmp_path / "mutant.c"
    c.write_text(mutated)
    so = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O1", "-fPIC", "-shared", "-std=c11", "-fopenmp", str(c), "-o", str(so), "-lm"],
                   check=True, capture_output=True)
    lib = oracle.load_library(str(so))
    failed = []
    for pin in pins.ALL_PINS:
        try:
            pin(lib)
        except AssertionError:
            failed.append(pin.__name__)
        except (ValueError, FloatingPointError):
            failed.append(pin.__name__)
    assert failed, f"mutant '{name}' passed every pin"
