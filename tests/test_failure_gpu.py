"""Failure detection without a GPU fault: the producer side of the
register-resident kernel (or of the tcgen05 kernel) withholds one hand-off (a flag nothing ever sets),
the consumer's bounded wait runs out after a short limit, the kernel stops
every role and reports KDA_ERR_DEVICE_TIMEOUT through the device status word,
and the context stays usable for the next launch."""
import ctypes

import pytest
import torch

from linear_attention_04_gb300 import kda as binding
from linear_attention_04_gb300 import kda_chunk_fwd, kda_device_status
from linear_attention_04_gb300.workloads import Workload, make_inputs

from parity import TOL, assert_close, f64, oracle_full

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("path", [binding.PATHS["mma"], binding.PATHS["mma_tc"], binding.PATHS["tc"]])
def test_withheld_handoff_reports_a_timeout_and_the_context_survives(path):
    w = Workload("fail", B=1, H=2, T=256, dk=128, dv=128, dtype=torch.bfloat16)
    inp = make_inputs(w, seed=404)
    g = {k_: (x.cuda() if isinstance(x, torch.Tensor) else x) for k_, x in inp.items()}
    out = torch.zeros((1, 256, 2, 128), device="cuda")
    fin = torch.zeros((1, 2, 128, 128), device="cuda")
    ws = torch.empty(256, dtype=torch.uint8, device="cuda")
    a = binding._Args(g["q"].data_ptr(), g["k"].data_ptr(), g["v"].data_ptr(),
                      g["theta"].data_ptr(), g["beta"].data_ptr(), -5.0, None, out.data_ptr(),
                      fin.data_ptr(), None, 1, 2, 256, 128, 128, 0, 1, path, 0)
    assert kda_device_status(clear=True) == 0
    lib = binding.load()
    rc = lib.kda_selftest_withheld_handoff(ctypes.byref(a), 50_000_000, ws.data_ptr(), ws.numel(),
                                           torch.cuda.current_stream().cuda_stream)
    assert rc == binding.KDA_OK
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == binding.KDA_ERR_DEVICE_TIMEOUT
    assert kda_device_status(clear=False) == 0
    # the next launch on the same context runs normally
    ro, rS = oracle_full(inp)
    o, S = kda_chunk_fwd(g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0)
    torch.cuda.synchronize()
    assert kda_device_status(clear=True) == 0
    assert_close(f64(o), ro, TOL[torch.bfloat16], "forward after the timeout")
    assert_close(f64(S), rS, TOL[torch.bfloat16], "state after the timeout")
