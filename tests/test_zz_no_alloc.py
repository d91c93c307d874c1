"""kda_chunk_fwd_segmented_noalloc (the segment-parallel forward over the
library's own scratch area) against the workspace entry point, on two
consecutive calls.  Collected last on purpose; passes alone as well."""
import pytest
import torch

from linear_attention_04_gb300 import kda as binding
from linear_attention_04_gb300 import kda_chunk_fwd_segmented, kda_device_status
from linear_attention_04_gb300.workloads import Workload, make_inputs

pytestmark = pytest.mark.gpu


def _inputs(seed):
    w = Workload("noalloc", B=1, H=6, T=5000, dk=128, dv=128, dtype=torch.bfloat16, init_std=0.03)
    return {k_: (x.cuda() if isinstance(x, torch.Tensor) else x)
            for k_, x in make_inputs(w, seed=seed).items()}


def test_noalloc_matches_workspace_entry_point_on_consecutive_calls():
    for call, seed in enumerate((11, 12)):
        g = _inputs(seed)
        args = (g["q"], g["k"], g["v"], g["theta"], g["beta"], -5.0, g["init_state"])
        ref_o, ref_S = kda_chunk_fwd_segmented(*args, segments=4)
        out = torch.empty_like(ref_o)
        fin = torch.empty_like(ref_S)
        binding.kda_chunk_fwd_segmented_noalloc(*args, out, fin, segments=4)
        torch.cuda.synchronize()
        assert kda_device_status(clear=True) == 0
        assert torch.equal(out, ref_o), f"call {call}: outputs differ"
        assert torch.equal(fin, ref_S), f"call {call}: final states differ"


def test_noalloc_rejects_a_call_larger_than_its_scratch():
    w = Workload("noalloc", B=1, H=32, T=65536, dk=128, dv=128, dtype=torch.bfloat16)
    g = {k_: (x.cuda() if isinstance(x, torch.Tensor) else x)
         for k_, x in make_inputs(w, seed=3).items()}
    out = torch.empty((1, 65536, 32, 128), device="cuda")
    with pytest.raises(binding.KdaError) as e:
        binding.kda_chunk_fwd_segmented_noalloc(g["q"], g["k"], g["v"], g["theta"], g["beta"],
                                                -5.0, None, out, None, segments=64)
    assert e.value.code == binding.KDA_ERR_SCRATCH_TOO_SMALL
