"""Long-context prefill: B=1, T=1,048,576, H=16, d=128, decay concentrated
near the bound, zero initial state.  The GPU runs all 16 heads in one call;
the fp64 oracle runs two of them over the whole million tokens and every
output and state element of those heads is compared."""
import pytest
import torch

from linear_attention_recurrence_fwd_gb300 import binding, build
from linear_attention_recurrence_fwd_gb300 import inputs as gen
from oracle import oracle as orc
from parity import assert_output_close, assert_state_close

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built(cuda_device):
    build.build()


def test_long_1m_two_heads_against_oracle():
    w = gen.WORKLOADS["long_1m"]
    dev = torch.device("cuda:0")
    x = gen.workload_inputs(w, device=dev)
    out, fin = binding.kda_chunk_fwd(x["q"], x["k"], x["v"], x["log_alpha"], x["beta"], None,
                                     out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert binding.kda_last_device_status() == 0
    heads = [0, 11]
    sub = {k: x[k][:, :, heads].cpu() for k in ("q", "k", "v", "log_alpha", "beta")}
    o = out[:, :, heads].cpu()
    s = fin[:, heads].cpu()
    del x, out, fin
    torch.cuda.empty_cache()
    ro, rs = orc.kda_recurrence(sub["q"], sub["k"], sub["v"], sub["log_alpha"], sub["beta"], None)
    assert_output_close(o, ro, what="long_1m")
    assert_state_close(s, rs, what="long_1m")
