"""The C ABI used from C alone: paged_fp8_kv_gk_gb300/examples/decode_step.c
(built here with the system C compiler against libgk.so and the CUDA runtime)
runs one decode step from raw input files, as append + attention or as the
two-launch step (gk_decode_step), with or without attention sinks; its output and group
buffers match the oracle (bf16 output within the parity tolerance, KV bytes
bit-exact)."""
import os
import shutil
import subprocess

import numpy as np
import pytest
import torch

import gk_inputs as gi
import gk_testlib as tl
import paged_fp8_kv_gk_gb300 as gk
from paged_fp8_kv_gk_gb300 import build as gkbuild

pytestmark = pytest.mark.gpu

CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


@pytest.fixture(scope="module")
def exe(tmp_path_factory):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    gk.lib()
    cc = shutil.which("cc") or shutil.which("gcc")
    if cc is None:
        pytest.skip("no C compiler")
    out = str(tmp_path_factory.mktemp("cexe") / "decode_step")
    src = os.path.join(gkbuild.HERE, "examples", "decode_step.c")
    subprocess.check_call([cc, "-O2", "-I", gkbuild.INCLUDE, "-I", os.path.join(CUDA, "include"),
                           src, "-o", out, "-L", gkbuild.BUILD_DIR, "-lgk",
                           "-L", os.path.join(CUDA, "lib64"), "-lcudart"])
    return out


def _write(d, name, a):
    np.ascontiguousarray(a).tofile(os.path.join(d, name))


def write_step_dir(d, name, with_sinks=False):
    """Write one step's inputs for the C program into directory d; returns
    (workload, control, step, cache, sinks or None)."""
    w = gi.get(name)
    c = gi.make_control(w)
    st = gi.make_step(w, "cpu")
    cache = gi.make_cache(w, c, "cpu")
    sh = gk.Shape.make(**gi.shape_dict(w, c))
    with open(os.path.join(d, "shape.bin"), "wb") as f:
        f.write(bytes(sh))
    for k in ("q", "k_new", "v_new"):
        _write(d, f"{k}.bin", gi.bf16_bits(st[k]))
    for k in ("cos", "sin", "k_scale", "v_scale"):
        _write(d, f"{k}.bin", np.asarray(getattr(c, k), np.float32))
    for k in ("bt_full", "bt_swa", "pos", "pos_w", "upd_full", "upd_swa"):
        _write(d, f"{k}.bin", np.asarray(getattr(c, k), np.int32))
    _write(d, "active.bin", np.asarray(c.active, np.uint8))
    for j, b in enumerate(cache):
        _write(d, f"cache_{j}.bin", b.numpy())
    sinks = gi.make_sinks(w) if with_sinks else None
    if sinks is not None:
        _write(d, "sinks.bin", sinks)
    return w, c, st, cache, sinks


@pytest.mark.parametrize("name,mode,with_sinks", [
    ("tiny", "split", False), ("gptoss_small", "split", False), ("block16_small", "split", False),
    ("gptoss_small", "fused", False), ("ragged_small", "fused", True),
    ("block16_small", "split", True)])
def test_c_program_step_matches_oracle(exe, tmp_path, name, mode, with_sinks):
    d = str(tmp_path)
    w, c, st, cache, sinks = write_step_dir(d, name, with_sinks)
    env = dict(os.environ)
    env["LD_LIBRARY_PATH"] = ":".join([gkbuild.BUILD_DIR, os.path.join(CUDA, "lib64"),
                                       env.get("LD_LIBRARY_PATH", "")])
    r = subprocess.run([exe, d, mode], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert mode in r.stdout
    ref, kb_ref, vb_ref = tl.oracle_step(w, c, st, cache, sinks=sinks)
    out_bits = np.fromfile(os.path.join(d, "out.bin"), np.uint16).reshape(ref.shape)
    out = (out_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    tl.check_out(out, None, ref, f"C program {name} {mode}")
    for j in range(len(cache)):
        got = np.fromfile(os.path.join(d, f"cache_out_{j}.bin"), np.uint8)
        half = got.size // 2
        assert np.array_equal(got[:half], kb_ref[j]) and np.array_equal(got[half:], vb_ref[j]), j
