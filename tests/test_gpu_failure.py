"""Failure detection on the GPU without a fault: a bounded wait that runs out.

With RA_TEST_WITHHOLD_V_TILE0=1 the attention kernel's TMA producer never
loads V tile 0.  The MMA issuer's mbarrier wait then expires (about two
seconds), the kernel records RA_ERR_DEVICE_TIMEOUT, the other roles leave
their loops, copies and MMAs already issued are drained, tensor memory is
freed and the kernel returns.  The host reads the code through
ra_get_device_status and the next normal call on the same context succeeds.
The test runs in a child process so the environment flag cannot leak into
other tests.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import sys, torch
sys.path.insert(0, sys.argv[1])
import __graft_entry__ as g
g.build()
import rope_causal_attention_gb300 as ra
import workloads as wl
Sq, Sk, Hq, Hkv, D = (int(a) for a in sys.argv[2:7])
q, k, v = [t.cuda() for t in wl.attn_qkv(1, Hq, Hkv, Sq, Sk, D, torch.bfloat16, 3)]
cos, sin = ra.make_tables(Sk, D, 10000.0)
ra.attn_fwd_causal_rope(q, k, v, cos, sin, kv_offset=Sk - Sq)
code = ra.ra_get_device_status()
print("STATUS", code)
import os
os.environ.pop("RA_TEST_WITHHOLD_V_TILE0")
o, lse = ra.attn_fwd_causal_rope(q, k, v, cos, sin, kv_offset=Sk - Sq)
print("AFTER", ra.ra_get_device_status(), bool(torch.isfinite(o.float()).all()))
"""


# one query tile (both slots of a block on it), three tiles of a grid that
# fits on the SMs (split blocks: the two slots share out the key tiles), and
# a grid past one wave (32 q / 8 kv heads, D = 128: 160 blocks of q-head
# pairs, every block running out its own wait)
@pytest.mark.parametrize("Sq,Sk,Hq,Hkv,D", [(128, 256, 2, 1, 64), (384, 512, 2, 1, 64),
                                            (1280, 1280, 32, 8, 128)])
def test_withheld_copy_times_out_cleanly(Sq, Sk, Hq, Hkv, D):
    env = dict(os.environ, RA_TEST_WITHHOLD_V_TILE0="1")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, str(Sq), str(Sk), str(Hq), str(Hkv),
                        str(D)], env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = dict(l.split(" ", 1) for l in r.stdout.splitlines() if l.startswith(("STATUS", "AFTER")))
    assert lines["STATUS"].strip() == "-6"          # RA_ERR_DEVICE_TIMEOUT
    assert lines["AFTER"].split() == ["0", "True"]  # context still usable
