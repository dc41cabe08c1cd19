"""The pins must bite: plant plausible mistakes in a copy of the oracle's C
source (on the CPU, in a temporary directory), build it, and check that the
oracle pin suite fails for every one of them."""
import os
import subprocess
import sys
import tempfile

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "zero_oracle.c")
PINS = ["tests/test_oracle_accounting.py", "tests/test_oracle_encodings.py",
        "tests/test_oracle_collectives.py", "tests/test_oracle_adam.py",
        "tests/test_oracle_steps.py", "tests/test_oracle_qgz.py", "tests/test_oracle_accum.py"]

# (name, text in the oracle source, planted replacement)
MUTATIONS = [
    ("no bias correction of m", "c->step_size = lr_sbc2 / bc1;", "c->step_size = lr_sbc2;"),
    ("no bias correction of v", "float sbc2 = sqrtf(bc2);", "float sbc2 = 1.0f;"),
    ("eps inside the root", "sqrtf(vi) + c->eps_hat", "sqrtf(vi + c->eps_hat)"),
    ("eps not bias-corrected", "c->eps_hat = hp->eps * sbc2;", "c->eps_hat = hp->eps;"),
    ("update sign flipped", "pi = pi - c->step_size * ratio;", "pi = pi + c->step_size * ratio;"),
    ("ratio transposed", "float ratio = mi / denom;", "float ratio = denom / (mi + 1e-30f);"),
    ("decay dropped", "pi = pi * c->decay;", "pi = pi;"),
    ("momentum uses 1-beta2", "c->omb1 * gi;", "c->omb2 * gi;"),
    ("variance of g, not g^2", "float g2 = gi * gi;", "float g2 = gi;"),
    ("beta1 power from beta2", "sc->beta1_pow * (double)hp->beta1;\n    sc->beta2_pow",
     "sc->beta1_pow * (double)hp->beta2;\n    sc->beta2_pow"),
    ("ranks summed in reverse", "for (int q = 0; q < n_d; ++q) sum", "for (int q = n_d - 1; q >= 0; --q) sum"),
    ("sum, not mean", "return rank_sum(n_d, grads, dtype, j) / divisor;", "return rank_sum(n_d, grads, dtype, j);"),
    ("loss scale ignored", "float scale = hp->loss_scaling ? sc->loss_scale : 1.0f;", "float scale = 1.0f;"),
    ("bf16 truncates", "return (uint16_t)shift_rne(u, 16);", "return (uint16_t)(u >> 16);"),
    ("fp16 subnormal off by one", "int s = 126 - e;", "int s = 127 - e;"),
    ("fp16 ties away from zero", "if (dropped > half || (dropped == half && (kept & 1))) kept += 1;",
     "if (dropped >= half) kept += 1;"),
    ("shard size floors", "long long per_rank = (psi + n_d - 1) / n_d;", "long long per_rank = psi / n_d + (psi % n_d > 1);"),
    # the first occurrence is the 16-bit gather
    ("gather at the wrong offset", "gathered[(long long)r * shard + i] = shards[r][i];",
     "gathered[(long long)r * len + i] = shards[r][i];"),
    ("clip always applied", "*applied = coef < 1.0f;", "*applied = 1;"),
    ("clip on the squared norm", "double norm = sqrt(sqnorm);", "double norm = sqnorm;"),
    ("overflow keeps the scale", "float half = sc->loss_scale * 0.5f;", "float half = sc->loss_scale;"),
    ("overflow advances t", "sc->good_steps = 0;\n    sc->overflow = 1;", "sc->good_steps = 0;\n    sc->overflow = 1;\n    sc->t += 1;"),
    ("quantizer divides by 128", "float s = amax / 127.0f;", "float s = amax / 128.0f;"),
    ("quantizer truncates", "q = rintf(zo_bf16_to_f32(x_bf16[i]) / s);", "q = truncf(zo_bf16_to_f32(x_bf16[i]) / s);"),
    ("stage 2 keeps full gradients", "    case 2:\n        grads = 2.0 * psi / n_d;", "    case 2:\n        grads = 2.0 * psi;"),
    ("qgZ scale of the wrong block", "const float* sblk = scales + ((long long)r * blocks_per_shard + i / block) * n_dp;",
     "const float* sblk = scales + ((long long)r * blocks_per_shard + (i + 1) / block) * n_dp;"),
    ("qgZ step ignores clipping",
     "zo_reduce_scatter_q(n_d, psi, S, block, codes, scales, divisor, shards);\n    return step_from_shards(n_d, psi, S, stage, shards, hp,",
     "zo_reduce_scatter_q(n_d, psi, S, block, codes, scales, divisor, shards);\n    zo_hparams nc = *hp;\n    nc.max_norm = 0.0f;\n    return step_from_shards(n_d, psi, S, stage, shards, &nc,"),
    ("qgZ ranks summed in reverse", "for (int q = 0; q < n_d; ++q) sum = sum + (float)codes[q][j] * sblk[q];",
     "for (int q = n_d - 1; q >= 0; --q) sum = sum + (float)codes[q][j] * sblk[q];"),
    ("qgZ blocks not aligned to shards",
     "long long off = (long long)r * shard + lo;\n                float* sc = scales +",
     "long long off = (long long)r * shard + lo + (r > 0);\n                float* sc = scales +"),
    ("accumulated step divides by n_d only", "float divisor = step_divisor(n_d * micro, hp, sc);",
     "float divisor = step_divisor(n_d, hp, sc);"),
    ("accumulated carry dropped at the step", "shards[j] = (carry + rank_sum(n_d, grads, grad_dtype, j)) / divisor;",
     "shards[j] = rank_sum(n_d, grads, grad_dtype, j) / divisor;"),
    ("accumulation ignores the accumulator", "float carry = acc_in ? acc_in[j] : 0.0f;", "float carry = 0.0f;"),
    ("accumulation continues one running sum", "acc_out[j] = carry + rank_sum(n_d, grads, dtype, j);",
     "for (int q = 0; q < n_d; ++q) carry = carry + zo_lp_to_f32(grads[q][j], dtype);\n        acc_out[j] = carry;"),
    ("stage 3 comm counts one gather", "return reduce_scatter + 2.0 * all_gather;", "return reduce_scatter + all_gather;"),
]


def _build(src_text, out_dir):
    c = os.path.join(out_dir, "zero_oracle.c")
    with open(c, "w") as f:
        f.write(src_text)
    with open(os.path.join(ROOT, "oracle", "zero_oracle.h")) as f:
        h = f.read()
    with open(os.path.join(out_dir, "zero_oracle.h"), "w") as f:
        f.write(h)
    lib = os.path.join(out_dir, "liboracle.so")
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC", "-shared", c, "-o", lib, "-lm"],
                   check=True, capture_output=True)
    return lib


def _pins_pass(lib):
    env = dict(os.environ, ZERO_ORACLE_LIB=lib)
    r = subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider",
                        "-m", "not gpu", *PINS], cwd=ROOT, env=env, capture_output=True, text=True)
    return r.returncode == 0


@pytest.fixture(scope="module")
def source():
    with open(SRC) as f:
        return f.read()


def test_unmutated_copy_passes(source):
    with tempfile.TemporaryDirectory() as d:
        assert _pins_pass(_build(source, d))


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(source, name, old, new):
    assert source.count(old) >= 1, "mutation anchor not found: " + name
    mutated = source.replace(old, new, 1)
    with tempfile.TemporaryDirectory() as d:
        assert not _pins_pass(_build(mutated, d)), "pins did not catch: " + name
