"""The oracle's pins catch plausible mistakes: each case plants one in a copy of the oracle.

A pin is only worth as much as the mistakes it would catch. Every case below edits a
copy of `oracle/` the way a slip in writing it could have (a wrong exponent bias, a
dropped term, a transposed index, a sign, an off-by-one), then runs the pin files
(`test_oracle_pins.py`, `test_indexer_oracle_pins.py`, and `test_workloads.py` for the
oracle's view of a seeded problem) against that copy in a child process and expects them
to fail. A control run of the unchanged copy must pass, and
each planted edit must match its source text exactly once, so a later change to the
oracle that moves the text makes this test fail rather than pass without planting
anything. CPU only; the repository's own files are never modified.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PIN_FILES = ("test_oracle_pins.py", "test_indexer_oracle_pins.py", "test_workloads.py")
SMLA = "smla_oracle.py"
IX = "indexer_oracle.py"
WO = "workload_oracle.py"

# (name, file, [(text, replacement), ...]): each edit is one plausible mistake.
MISTAKES = [
    # E4M3FN decode / encode (OCP 8-bit floating point formats)
    ("e4m3 exponent bias 8", SMLA, [("np.ldexp(1.0 + m / 8.0, e - 7)", "np.ldexp(1.0 + m / 8.0, e - 8)")]),
    ("e4m3 subnormal exponent -7", SMLA, [("np.ldexp(m / 8.0, -6)", "np.ldexp(m / 8.0, -7)")]),
    ("e4m3 whole top binade NaN", SMLA, [("(e == 15) & (m == 7)", "(e == 15)")]),
    ("e4m3 sign ignored", SMLA, [("val = np.where(s == 1, -mag, mag)", "val = mag")]),
    ("encode ties to odd", SMLA, [("(hi % 2 == 0)", "(hi % 2 == 1)")]),
    ("encode ties away from zero", SMLA, [("((d_hi == d_lo) & (hi % 2 == 0))", "(d_hi == d_lo)")]),
    ("encode drops negative zero", SMLA, [("code | np.where(neg, 0x80, 0)", "code | np.where(neg & (a > 0), 0x80, 0)")]),
    ("encode truncates", SMLA, [("take_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))",
                                 "take_hi = d_hi == 0")]),
    ("bf16 bits read as the low half", SMLA, [("astype(np.uint32) << np.uint32(16)", "astype(np.uint32) << np.uint32(15)")]),
    # fp8_ds block scales and the 656-byte row
    ("pow2 scale rounded down", SMLA, [("np.where(m == 0.5, v, np.ldexp(1.0, e))", "np.where(m == 0.5, v, np.ldexp(1.0, e - 1))")]),
    ("scale from the E4M3FNUZ maximum 240", SMLA, [("ratio = f32(amax / E4M3_MAX)", "ratio = f32(amax / 240.0)")]),
    ("scale blocks strided instead of contiguous", SMLA,
     [("latent.reshape(latent.shape[0], 4, BLOCK)).max(axis=2)", "latent.reshape(latent.shape[0], BLOCK, 4)).max(axis=1)")]),
    ("zero block scale 0", SMLA, [("return np.where(amax == 0, 1.0, sc)", "return np.where(amax == 0, 0.0, sc)")]),
    ("packer multiplies by the scale", SMLA, [("q = f32(lat / np.repeat(sc, BLOCK, axis=1))", "q = f32(lat * np.repeat(sc, BLOCK, axis=1))")]),
    ("RoPE stored before the scales", SMLA,
     [("out[:, LATENT:LATENT + 16] = sc", "out[:, LATENT + 128:] = sc"),
      ("out[:, LATENT + 16:] = np.asarray(rope_bits", "out[:, LATENT:LATENT + 128] = np.asarray(rope_bits")]),
    ("scales stored big-endian", SMLA, [('sc.astype("<f4")', 'sc.astype(">f4")')]),
    ("per-tensor packer multiplies by kv_scale", SMLA,
     [("q = f32(x / float(f32(kv_scale)))", "q = f32(x * float(f32(kv_scale)))")]),
    ("per-tensor packer leaves RoPE out", SMLA,
     [("x = np.concatenate([lat, rope], axis=1)", "x = np.concatenate([lat, 0 * rope], axis=1)")]),
    ("bf16 row with RoPE first", SMLA,
     [("row = np.concatenate([np.asarray(latent_bits, dtype=\"<u2\").reshape(n, LATENT),\n"
       "                          np.asarray(rope_bits, dtype=\"<u2\").reshape(n, ROPE)], axis=1)",
       "row = np.concatenate([np.asarray(rope_bits, dtype=\"<u2\").reshape(n, ROPE),\n"
       "                          np.asarray(latent_bits, dtype=\"<u2\").reshape(n, LATENT)], axis=1)")]),
    # dequantisation
    ("dequant scale of dim d taken as d % 4", SMLA,
     [("lat = f32(e4m3_decode(codes) * np.repeat(sc, BLOCK, axis=1))", "lat = f32(e4m3_decode(codes) * np.tile(sc, BLOCK))")]),
    ("dequant product not rounded to fp32", SMLA,
     [("lat = f32(e4m3_decode(codes) * np.repeat(sc, BLOCK, axis=1))", "lat = e4m3_decode(codes) * np.repeat(sc, BLOCK, axis=1)")]),
    ("dequant of per-tensor rows drops kv_scale", SMLA,
     [("return f32(e4m3_decode(rows[:, :DIM]) * float(f32(kv_scale)))", "return f32(e4m3_decode(rows[:, :DIM]))")]),
    ("dequant reads the RoPE from the scale bytes", SMLA,
     [("rope = bf16_bits_to_f64(rows[:, LATENT + 16:]", "rope = bf16_bits_to_f64(rows[:, LATENT:LATENT + 128]")]),
    # addressing
    ("request of token t is t mod next_n", SMLA, [("return t // next_n", "return t % next_n")]),
    ("req_id_per_token ignored", SMLA, [("if req_id_per_token is not None:\n        return int(req_id_per_token[t])",
                                         "if False:\n        return int(req_id_per_token[t])")]),
    ("page looked up by idx mod P", SMLA, [("page = int(pt_row[idx // page_size])", "page = int(pt_row[idx % page_size])")]),
    ("in-page offset idx // P", SMLA, [("phys.append(page * page_size + idx % page_size)", "phys.append(page * page_size + idx // page_size)")]),
    ("page table skipped", SMLA, [("phys.append(page * page_size + idx % page_size)", "phys.append(idx)")]),
    ("padding counted as invalid", SMLA, [("if idx == -1:\n            continue", "if idx == -1:\n            n_invalid += 1\n            continue")]),
    ("out-of-range page entries kept", SMLA, [("if page < 0 or page >= num_pages:", "if page < 0:")]),
    ("decode takes the token as its request", SMLA,
     [("        r = request_of_token(t, next_n, req_id_per_token)\n        _, phys,", "        r = t\n        _, phys,")]),
    # attention
    ("softmax scale dropped", SMLA, [("s = float(sm_scale) * (q @ keys.T)", "s = (q @ keys.T)")]),
    ("scores from the latent only", SMLA, [("s = float(sm_scale) * (q @ keys.T)", "s = float(sm_scale) * (q[:, :LATENT] @ keys[:, :LATENT].T)")]),
    ("values are the last 512 dims", SMLA, [("out = (e @ keys[:, :LATENT])", "out = (e @ keys[:, -LATENT:])")]),
    ("sink dropped from the denominator", SMLA, [("denom = denom + np.exp(sig - m[:, 0])", "denom = denom")]),
    ("sink not shifted by the running max", SMLA, [("denom = denom + np.exp(sig - m[:, 0])", "denom = denom + np.exp(sig)")]),
    ("sink weighted like a score", SMLA, [("denom = denom + np.exp(sig - m[:, 0])", "denom = denom + np.exp(sm_scale * sig - m[:, 0])")]),
    ("lse in base 2", SMLA, [("lse = m[:, 0] + np.log(denom)", "lse = m[:, 0] + np.log2(denom)")]),
    ("lse leaves the sink out", SMLA, [("lse = m[:, 0] + np.log(denom)", "lse = lse0.copy()")]),
    ("lse without sink taken with the sink", SMLA,
     [("lse0 = m0 + np.log(np.exp(s - m0[:, None]).sum(axis=1))", "lse0 = m[:, 0] + np.log(denom + (0.0 if sig is None else np.exp(sig - m[:, 0])))")]),
    ("empty selection with a sink gives -inf", SMLA, [("lse = lse0.copy() if sig is None else sig.copy()", "lse = lse0.copy()")]),
    ("FP8 q ignores q_scale", SMLA, [("return e4m3_decode(q) * float(np.float32(q_scale))", "return e4m3_decode(q)")]),
    # fused store: norm, rotation, bf16 rounding
    ("bf16 rounding truncates", SMLA, [("np.rint(m * 256.0)", "np.trunc(m * 256.0)")]),
    ("bf16 rounding keeps 9 bits", SMLA, [("np.ldexp(np.rint(m * 256.0), e - 8)", "np.ldexp(np.rint(m * 512.0), e - 9)")]),
    ("norm without eps", SMLA, [("+ float(np.float32(eps)))", ")")]),
    ("norm by the sum of squares", SMLA, [("(x * x).mean(axis=1, keepdims=True)", "(x * x).sum(axis=1, keepdims=True)")]),
    ("norm without the weight", SMLA, [("bf16_rne(x * r * w[None, :])", "bf16_rne(x * r)")]),
    ("norm without the square root", SMLA, [("r = 1.0 / np.sqrt(", "r = 1.0 / (")]),
    ("rotation by minus the angle", SMLA,
     [("out[:, 0::2] = a * c - b * s", "out[:, 0::2] = a * c + b * s"),
      ("out[:, 1::2] = a * s + b * c", "out[:, 1::2] = -a * s + b * c")]),
    ("rotation pairs the two halves", SMLA,
     [("a, b = r[:, 0::2], r[:, 1::2]", "a, b = r[:, :32], r[:, 32:]"),
      ("out[:, 0::2] = a * c - b * s", "out[:, :32] = a * c - b * s"),
      ("out[:, 1::2] = a * s + b * c", "out[:, 32:] = a * s + b * c")]),
    ("store skips the rotation", SMLA, [("rope = f64_to_bf16_bits(rope_bf16(rope_bits, cos, sin))", "rope = rope_bits")]),
    ("store skips the norm", SMLA, [("lat = f64_to_bf16_bits(rms_norm_bf16(latent_bits, weight_bits, eps))", "lat = latent_bits")]),
    # indexer logits and top-k
    ("visible prefix one slot short", IX, [("int(ctx) - int(next_n) + 1 + int(i)", "int(ctx) - int(next_n) + int(i)")]),
    ("visible prefix the same for every row", IX, [("int(ctx) - int(next_n) + 1 + int(i)", "int(ctx)")]),
    ("page's scales read before its codes", IX,
     [("codes = cache_page[:page_size * INDEX_DIM]", "codes = cache_page[page_size * 4:page_size * (INDEX_DIM + 4)]"),
      ("scales = cache_page[page_size * INDEX_DIM:page_size * (INDEX_DIM + 4)]", "scales = cache_page[:page_size * 4]")]),
    ("index slot's page by s mod P", IX, [("cache[int(pt_row[s0 // page_size])]", "cache[int(pt_row[s0 % page_size])]")]),
    ("logits without the ReLU", IX, [("act = np.maximum(0.0, dots * scales[None, :])", "act = dots * scales[None, :]")]),
    ("logits without the key scale", IX, [("act = np.maximum(0.0, dots * scales[None, :])", "act = np.maximum(0.0, dots)")]),
    ("logits without the head weights", IX, [("return np.asarray(weights, dtype=np.float64) @ act", "return act.sum(axis=0)")]),
    ("ReLU after the sum over heads", IX,
     [("act = np.maximum(0.0, dots * scales[None, :])\n    return np.asarray(weights, dtype=np.float64) @ act",
       "act = dots * scales[None, :]\n    return np.maximum(0.0, np.asarray(weights, dtype=np.float64) @ act)")]),
    ("token's request row from the wrong end", IX, [("r, i = divmod(int(t), next_n)", "r, i = divmod(int(t), next_n)\n        i = next_n - 1 - i")]),
    ("top-k takes the smallest", IX, [('order = np.argsort(-logits, kind="stable")', 'order = np.argsort(logits, kind="stable")')]),
    ("top-k one short", IX, [("return np.sort(order[:k])", "return np.sort(order[:k - 1])")]),
    ("top-k ties to the highest index", IX, [('order = np.argsort(-logits, kind="stable")',
                                              'order = n - 1 - np.argsort(-logits[::-1], kind="stable")')]),
    # the oracle's view of a seeded problem's cache
    ("cache row one slot along", WO, [("return self.rows[loc * self.P + phys % self.P]",
                                       "return self.rows[loc * self.P + (phys + 1) % self.P]")]),
    ("cache packed with fp32 scales", WO, [("O.pack_fp8_ds(_bits(lat), _bits(rope), scale_mode)",
                                            "O.pack_fp8_ds(_bits(lat), _bits(rope), O.SCALE_FP32)")]),
]


def _copy_tree(dst: str, file_name: str | None = None, edits=()):
    """Copy the oracle package and the pin files under dst, planting edits in file_name."""
    for pkg in ("oracle", "workloads"):
        shutil.copytree(os.path.join(ROOT, pkg), os.path.join(dst, pkg), ignore=shutil.ignore_patterns("__pycache__"))
    os.makedirs(os.path.join(dst, "tests"))
    for f in ("conftest.py",) + PIN_FILES:
        shutil.copy(os.path.join(ROOT, "tests", f), os.path.join(dst, "tests", f))
    if file_name is None:
        return
    path = os.path.join(dst, "oracle", file_name)
    with open(path) as fh:
        src = fh.read()
    for text, repl in edits:
        assert src.count(text) == 1, f"{file_name}: the text to edit is not found once: {text!r}"
        src = src.replace(text, repl)
    with open(path, "w") as fh:
        fh.write(src)


def _env():
    env = {k: v for k, v in os.environ.items() if k != "PYTHONPATH"}
    env["PYTHONDONTWRITEBYTECODE"] = "1"
    env["CUDA_VISIBLE_DEVICES"] = ""
    env["OMP_NUM_THREADS"] = "1"  # the children run side by side; one thread each
    return env


def _run_pins(dst: str) -> subprocess.CompletedProcess:
    return subprocess.run(
        [sys.executable, "-m", "pytest", "-x", "-q", "-p", "no:cacheprovider", "-m", "not gpu",
         *[os.path.join("tests", f) for f in PIN_FILES]],
        cwd=dst, env=_env(), capture_output=True, text=True, timeout=600)


def test_control_copy_passes_and_is_the_one_imported(tmp_path):
    dst = str(tmp_path / "control")
    _copy_tree(dst)
    where = subprocess.run([sys.executable, "-c", "import oracle; print(oracle.__file__)"],
                           cwd=dst, env=_env(), capture_output=True, text=True, timeout=300)
    assert where.returncode == 0, where.stderr
    assert os.path.realpath(where.stdout.strip()).startswith(os.path.realpath(dst))
    r = _run_pins(dst)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-2000:]


def test_pins_catch_every_planted_mistake(tmp_path):
    dirs = []
    for k, (name, file_name, edits) in enumerate(MISTAKES):
        dst = str(tmp_path / f"m{k:02d}")
        _copy_tree(dst, file_name, edits)
        dirs.append((name, dst))
    with ThreadPoolExecutor(max_workers=max(1, min(8, os.cpu_count() or 1))) as pool:
        results = list(pool.map(lambda nd: (nd[0], _run_pins(nd[1])), dirs))
    survived = [name for name, r in results if r.returncode == 0]
    assert not survived, f"no pin fails when the oracle has these mistakes: {survived}"
    # a failure must come from a pin, not from a crash of the test run itself
    broken = [name for name, r in results if r.returncode not in (1,)]
    assert not broken, f"the pin run did not complete for: {broken}"

