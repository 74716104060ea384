"""Failure handling on the GPU without a fault: a bounded wait that runs out ends as a status
word the host reads, the context stays usable, and the compute calls do no work while the
status word is set."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
import chunked_gated_linear_gb300 as gcl  # noqa: E402
from chunked_gated_linear_gb300 import synth  # noqa: E402
from gpu_util import CANARY, DEV, Meta, check_fwd, run_fwd, to_device  # noqa: E402

GCL_DEV_WAIT_TIMEOUT = 5


def test_wait_limit_sets_status_and_blocks_later_work():
    status = torch.zeros(1, dtype=torch.int32, device=DEV)
    gcl.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == GCL_DEV_WAIT_TIMEOUT
    # the compute kernels read the status word first and leave every output untouched
    w = synth.varlen("timeout", synth.GDN, "bf16", [100, 30], 2, 160, 2, 128, 128, seed=71)
    x = synth.make_inputs(w)
    d = to_device(w, x)
    meta = Meta(w.t_max, w.n_max)
    meta.build(d["cu_seqlens"])
    torch.cuda.synchronize()
    meta.status.fill_(GCL_DEV_WAIT_TIMEOUT)
    out = run_fwd(w, d, meta=meta)
    torch.cuda.synchronize()
    assert (out["o"].float().cpu().numpy() == np.float32(CANARY)).all()
    assert (out["ht"].cpu().numpy() == np.float32(CANARY)).all()
    # the context is still usable: a fresh status word and the same call give the oracle's result
    out = run_fwd(w, d)
    check_fwd(w, x, out, label="after the timeout")


def test_wait_limit_keeps_a_set_status():
    """A status word that already holds an error keeps it (the first failure is reported)."""
    status = torch.full((1,), 3, dtype=torch.int32, device=DEV)
    gcl.selftest_wait_timeout(status)
    torch.cuda.synchronize()
    assert int(status.item()) == 3
