"""Device-side failure detection on the GPU, without a fault: a bounded wait
that nothing satisfies runs out, the kernel records RA_ERR_DEVICE_TIMEOUT and
returns, ra_device_status reports it once, and the context stays usable."""
import pytest
import torch

import ring_context_parallelism_gb300 as ra
from ring_context_parallelism_gb300 import ra as rab
from ring_context_parallelism_gb300.inputs import WORKLOADS, attention_inputs, small

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from ring_context_parallelism_gb300.build import build
    build()
    ra.load()


def test_bounded_wait_runs_out_and_is_reported():
    ra.selftest_wait_timeout(50_000_000)          # 50 ms
    with pytest.raises(ra.RAError) as e:
        ra.device_status()
    assert e.value.status == rab.RA_ERR_DEVICE_TIMEOUT
    ra.device_status()                            # reported once, then cleared
    # the context still runs the attention path
    w = small(WORKLOADS["gqa_causal_prefill_32k"], S=512, n_shards=2, Hq=2, Hkv=1, seed=1)
    q, k, v = (t.cuda() for t in attention_inputs(w, "cpu"))
    O, L = ra.attn(q, k, v, w.n_shards, w.block, True)
    ra.device_status()
    assert torch.isfinite(O.float()).all() and torch.isfinite(L).all()
