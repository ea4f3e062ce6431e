"""Parity run of the fp32-FMA comparison path of the attention kernel (the
library picks it when GK_ATTN_PATH=fma is set before its first call, so this
runs in its own process): small workloads, with and without attention sinks,
against the oracle at the parity tolerance.  Exit status 0 on success."""
import os
import sys

import numpy as np
import torch

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))

import gk_inputs as gi  # noqa: E402
import gk_testlib as tl  # noqa: E402
import paged_fp8_kv_gk_gb300 as gk  # noqa: E402


def main() -> int:
    assert os.environ.get("GK_ATTN_PATH") == "fma"
    for name in ("gptoss_small", "long_small", "swa_small_peaky"):
        w = gi.get(name)
        c = gi.make_control(w)
        st = gi.make_step(w, "cpu")
        cache = gi.make_cache(w, c, "cpu")
        for sinks in (None, gi.make_sinks(w)):
            ref, kb_ref, vb_ref = tl.oracle_step(w, c, st, cache, sinks=sinks)
            g = tl.GpuStep(w, c, st, cache, sinks=sinks)
            g.append()
            g.attention()
            torch.cuda.synchronize()
            assert gk.gk_read_device_error() == 0
            for j in range(len(g.cache)):
                assert np.array_equal(g.cache[j][0].cpu().numpy().reshape(-1), kb_ref[j])
            tl.check_out(g.out.float().cpu().numpy().astype(np.float64),
                         g.out_f32.cpu().numpy().astype(np.float64), ref,
                         f"fma {name} sinks={sinks is not None}")
    print("fma path ok")
    return 0


if __name__ == "__main__":
    sys.exit(main())
