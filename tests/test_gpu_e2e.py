"""The benchmark's end-to-end prefill (bench.E2EPipeline: inputs packed in one pinned host buffer,
two device buffer sets, upload / compute / download on three streams) delivers exactly what a direct
kda_forward call on device inputs computes, for every step of the stream of requests."""
import sys

import pytest
import torch

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from linear_attention_recurrence_kda_gb300 import binding as B  # noqa: E402
from linear_attention_recurrence_kda_gb300 import inputs as I  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("wid,lengths", [(1, None), (2, [700, 0, 333, 1500, 17])], ids=["prefill-4096", "varlen"])
def test_e2e_pipeline_outputs_equal_a_direct_call(wid, lengths):
    dev = torch.device("cuda")
    d = bench.device_workload(I, wid, dev, lengths=lengths)
    ref_o, ref_s = B.kda_forward(d["q"], d["k"], d["v"], d["z"], d["A"], d["beta"], initial_state=d["S0"],
                                 cu_seqlens=d["cu_seqlens"], max_seqlen=max(d["lengths"]))
    torch.cuda.synchronize()
    pipe = bench.E2EPipeline(B, d, dev)
    for i in range(5):  # odd and even steps: both device buffer sets, reused after their outputs left
        pipe.step()
        torch.cuda.synchronize()
        o, s = pipe.outputs()
        assert torch.equal(o, ref_o.cpu()), f"step {i}: outputs differ from the direct call"
        assert torch.equal(s, ref_s.cpu()), f"step {i}: final states differ from the direct call"
    # and back to back without synchronising between steps: the last step's results
    for _ in range(4):
        pipe.step()
    torch.cuda.synchronize()
    o, s = pipe.outputs()
    assert torch.equal(o, ref_o.cpu()) and torch.equal(s, ref_s.cpu())
    assert pipe.h2d_bytes >= sum(d[k].numel() * d[k].element_size() for k in pipe.KEYS)
