"""Failure detection on the GPU without a fault: a bounded wait that runs out.

Every wait inside the decode kernels is bounded by wall time
(PA_WAIT_TIMEOUT_MS).  The test hook PA_OPT_DROP_FIRST_FILL makes every
decode CTA leave its first pipeline stage unfilled -- a phase that nothing
completes -- so the consumers' wait runs out.  The kernel must then record
PA_DEVERR_TIMEOUT, drain its copies and return; the host reads
PA_ERR_DEVICE_TIMEOUT, and the same context keeps working.  Runs in a child
process because the wait limit is read once per process.
"""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent("""
    import os, sys, time
    sys.path.insert(0, {root!r})
    import torch
    from paged_kv_cache_132_gb300 import api, native, workloads
    native.load()
    for kernel in ("mma", "simt"):
        api.set_option("decode_kernel_simt", kernel == "simt")
        w = workloads.make("llama8b", device="cuda", num_seqs=16)
        k, v = w.k_cache.clone(), w.v_cache.clone()
        api.reshape_and_cache(w.new_key, w.new_value, k, v, w.slot_mapping)
        mc = int(w.context_lens.max())
        run = lambda: api.decode(w.query, k, v, w.block_tables, w.context_lens, w.scale, max_context_len=mc)
        ref = run()
        assert api.get_device_error() == (0, 0)
        api.set_option("drop_first_fill", True)
        t0 = time.time()
        run()
        status, code = api.get_device_error()
        elapsed = time.time() - t0
        api.set_option("drop_first_fill", False)
        assert status == -6 and code & 0x10, (status, code)
        assert elapsed < 20.0, elapsed
        again = run()
        assert api.get_device_error() == (0, 0)
        assert torch.max(torch.abs(again - ref)).item() <= 1e-6
        print(kernel, "timeout-detected", round(elapsed, 3), flush=True)
""")


def test_bounded_wait_runs_out_and_context_survives():
    env = dict(os.environ, PA_WAIT_TIMEOUT_MS="200")
    env.pop("PA_DEBUG_DROP_FIRST_FILL", None)
    env.pop("PA_DECODE_KERNEL", None)
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env, cwd=ROOT, timeout=300,
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.count("timeout-detected") == 2, r.stdout
