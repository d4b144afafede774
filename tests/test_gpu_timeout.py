"""The bounded waits end in an error status, not a hang: with the test hook
BDSA_TEST_EXPIRE_OWNER_WAITS=1 the owner merge of the attention (64-row and
128-row tiles) waits for a ticket that no CTA publishes, gives up after the
wait limit (1 s) and the call's dev_status reads BDSA_DEVICE_TIMEOUT (17).
The same process then runs the call again without the hook: status 0 and the
oracle's output, so the context stays usable.  Run in a child process so that
the hook cannot leak into other tests."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent("""
    import dataclasses, os, sys
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    sys.path.insert(0, ROOT)
    import numpy as np, torch
    import block_diffusion_speculative_attn_gb300 as bdsa
    from block_diffusion_speculative_attn_gb300 import workloads as wl
    from gpu_helpers import DevAttn, run_attn, oracle_attn_requests, assert_attn_close
    # four requests of 2500-3000 keys over the whole GPU: every unit is cut
    # between CTAs (Qwen3-8B shape: G * B = 64; LLaDA2.0-style: 128)
    cfg = dataclasses.replace(wl.config(NAME), bs=4, ctx=((2500, 3000),))
    d = DevAttn(wl.make_attn_inputs(cfg, device="cpu", seed=3))
    os.environ["BDSA_TEST_EXPIRE_OWNER_WAITS"] = "1"
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    run_attn(d, bdsa.VERIFY, status=st)
    assert st.item() == 17, st.item()
    del os.environ["BDSA_TEST_EXPIRE_OWNER_WAITS"]
    st.zero_()
    out, lse = run_attn(d, bdsa.VERIFY, status=st)
    assert st.item() == 0, st.item()
    ref, ref_lse, rows = oracle_attn_requests(d, [0, 3], bdsa.VERIFY)
    assert_attn_close(out[torch.from_numpy(rows).cuda()], ref, lse[torch.from_numpy(rows).cuda()],
                      ref_lse, tag="after the expired waits")
    print("ok")
""")


@pytest.mark.parametrize("name", ["qwen3_8b_verify", "llada2_block_draft"],
                         ids=["rows64", "rows128"])
def test_owner_merge_wait_expires_with_timeout_status(name):
    env = dict(os.environ)
    env.pop("BDSA_TEST_EXPIRE_OWNER_WAITS", None)
    head = f"ROOT = {ROOT!r}\nNAME = {name!r}\n"
    r = subprocess.run([sys.executable, "-c", head + CHILD], env=env, cwd=ROOT,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
