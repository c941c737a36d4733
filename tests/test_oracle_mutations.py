"""The oracle's pins catch plausible mistakes in it.

Each case plants one mistake in a temporary copy of the oracle (its C half or its
numpy half), on the CPU, and runs the pins it names against that copy in a child
process: at least one of them must fail.  A copy with nothing planted passes every
pin named here, so a failure comes from the planted mistake, not from the copying.
The children run at once, each with two OpenMP threads.
"""
import os
import shutil
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PINS = os.path.join(ROOT, "tests", "test_oracle_pins.py")

# (name, file under oracle/, text as it stands, text planted in its place, pins (-k))
MUTATIONS = [
    # page table and storage
    ("slot of a token one off", "pkv_oracle.c",
     "int64_t slot = t % c->page_size;", "int64_t slot = (t + 1) % c->page_size;", "worked_example"),
    ("kv_len one short", "pkv_oracle.c",
     "return (n - 1) * c->page_size + c->kv_last_page_len[b];",
     "return (n - 1) * c->page_size + c->kv_last_page_len[b] - 1;", "worked_example or matches_sdpa"),
    ("fp16 subnormal scale", "pkv_oracle.c",
     "ldexp((double)m, -24)", "ldexp((double)m, -25)", "decode16"),
    ("bf16 taken from the wrong half", "pkv_oracle.c",
     "(uint32_t)b << 16", "(uint32_t)b << 15", "decode16"),
    # attention
    ("causal limit one off", "pkv_oracle.c",
     "causal ? i + kv_len - qo_len + 1 : kv_len", "causal ? i + kv_len - qo_len : kv_len", "causal_row_sees"),
    ("query head to kv head map", "pkv_oracle.c",
     "int kvh = h / group;", "int kvh = h % num_kv_heads;", "matches_sdpa"),
    ("owner of a query row", "pkv_oracle.c",
     "if (qo_indptr[mid] <= r)", "if (qo_indptr[mid] < r)", "matches_sdpa"),
    ("soft-cap before the scale", "pkv_oracle.c",
     "logit = logits_cap * tanh(logit / logits_cap);",
     "logit = sm_scale * logits_cap * tanh(dot / logits_cap);", "softcap"),
    ("K read in place of V", "pkv_oracle.c",
     "token_row(&c, b, t, 1, kvh)", "token_row(&c, b, t, 0, kvh)", "uniform_v"),
    ("lse in base 2", "pkv_oracle.c",
     "double l = mx + log(sum);", "double l = mx + log2(sum);", "lse_matches_scipy or zero_query"),
    ("empty key set gives lse 0", "pkv_oracle.c",
     "*lrow = -INFINITY;", "*lrow = 0.0;", "empty_request"),
    ("mask bits most significant first", "pkv_oracle.c",
     "(mask[bit >> 3] >> (bit & 7))", "(mask[bit >> 3] >> (7 - (bit & 7)))", "custom_mask"),
    ("mask row stride of qo_len", "pkv_oracle.c",
     "mask_off[b] + i * kv_len + t", "mask_off[b] + i * qo_len + t", "custom_mask"),
    # merge_state and cascade
    ("merge weight against the max", "pkv_oracle.c",
     "double w = exp(lse[k * n + r] - l);", "double w = exp(lse[k * n + r] - m);", "merge"),
    ("cascade drops its last level", "__init__.py",
     "states = [attention_of(b, threads=threads) for b in level_batches]",
     "states = [attention_of(b, threads=threads) for b in level_batches[:max(1, len(level_batches) - 1)]]",
     "cascade"),
    # append stage
    ("RoPE turns the other way", "__init__.py",
     "[a * c - b * s, b * c + a * s]", "[a * c + b * s, b * c - a * s]", "rope"),
    ("RoPE pairs neighbours", "__init__.py",
     "a, b = xv[..., :half], xv[..., half:]", "a, b = xv[..., 0::2], xv[..., 1::2]", "rope"),
    ("RoPE frequency exponent", "__init__.py",
     "-2.0 * np.arange(half, dtype=np.float64) / d", "-1.0 * np.arange(half, dtype=np.float64) / d", "rope"),
    ("append one position early", "__init__.py",
     "p = kv_len - n_new + i", "p = kv_len - n_new + i - 1", "append"),
    ("append rotates the values", "__init__.py",
     "v = decode16(v_new)", "v = rope(v_new, pos, rope_theta) if rope_theta > 0 else decode16(v_new)",
     "append_then_gather"),
    ("rounding ties away from zero", "__init__.py",
     "np.rint(np.ldexp(x[fin], -ulp_exp))", "np.trunc(np.ldexp(x[fin], -ulp_exp) + np.copysign(0.5, x[fin]))",
     "encode16"),
    ("overflow a full ulp past the top", "__init__.py",
     "max_finite + top_ulp / 2", "max_finite + top_ulp", "encode16"),
]

_CHILD = textwrap.dedent("""
    import sys
    copy, root, pins, expr = sys.argv[1:5]
    sys.path.insert(0, copy)
    sys.path.insert(1, root)
    import oracle
    if not oracle.__file__.startswith(copy):
        sys.exit(90)
    oracle.build(force=True)
    import pytest
    sys.exit(pytest.main([pins, "-q", "-x", "-k", expr, "-p", "no:cacheprovider", "--rootdir", root]))
""")


def _copy_oracle(dst, mutation=None):
    shutil.copytree(os.path.join(ROOT, "oracle"), os.path.join(dst, "oracle"),
                    ignore=shutil.ignore_patterns("_build", "__pycache__"))
    if mutation is not None:
        _, fname, old, new, _ = mutation
        path = os.path.join(dst, "oracle", fname)
        with open(path) as f:
            src = f.read()
        assert src.count(old) == 1, f"{fname} no longer holds exactly one {old!r}"
        with open(path, "w") as f:
            f.write(src.replace(old, new))


@pytest.fixture(scope="module")
def outcomes(tmp_path_factory):
    """(exit code, output) of the pins, per mutation name and for the clean copy."""
    union = " or ".join(f"({m[4]})" for m in MUTATIONS)
    jobs = [("clean copy", None, union)] + [(m[0], m, m[4]) for m in MUTATIONS]
    env = dict(os.environ, OMP_NUM_THREADS="2", PYTHONDONTWRITEBYTECODE="1")
    procs = {}
    for name, mut, expr in jobs:
        d = str(tmp_path_factory.mktemp("mut"))
        _copy_oracle(d, mut)
        procs[name] = subprocess.Popen([sys.executable, "-c", _CHILD, d, ROOT, PINS, expr], cwd=d, env=env,
                                       stdout=subprocess.PIPE, stderr=subprocess.STDOUT, text=True)
    out = {}
    for name, p in procs.items():
        try:
            text, _ = p.communicate(timeout=600)
        except subprocess.TimeoutExpired:
            p.kill()
            text, _ = p.communicate()
        out[name] = (p.returncode, text)
    return out


def test_clean_copy_passes_every_named_pin(outcomes):
    code, text = outcomes["clean copy"]
    assert code == 0, text[-3000:]


@pytest.mark.parametrize("mutation", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_fails_a_pin(outcomes, mutation):
    code, text = outcomes[mutation[0]]
    # 1: pins ran and one failed; 90: the copy was not the oracle imported;
    # 2-5: interrupted, internal error, usage error, nothing selected
    assert code == 1, f"exit {code}:\n{text[-3000:]}"
    assert " failed" in text, text[-3000:]
