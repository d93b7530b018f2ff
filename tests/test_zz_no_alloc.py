"""kda_chunk_prefill_noalloc (record ring in the library's static device scratch) against
the workspace entry point kda_chunk_prefill_ws: two calls in a row, identical results.

Kept in a file of its own, collected last, so that it runs after everything else too."""
import pytest
import torch

from kimi_delta_attention_09_gb300 import inputs
from _helpers import cuda

pytestmark = pytest.mark.gpu


def _run(case, entry, out_dtype=torch.float32):
    from kimi_delta_attention_09_gb300 import _native
    q, k, v, g, beta = (cuda(x) for x in (case.q, case.k, case.v, case.g, case.beta))
    cu = cuda(case.cu_seqlens)
    out = torch.full(v.shape, float("nan"), dtype=out_dtype, device="cuda")
    fin = torch.full((case.N, case.H, case.K, case.V), float("nan"), device="cuda")
    if entry == "ws":
        n = _native.kda_chunk_prefill_workspace_bytes(case.N, case.H, case.K, case.V, case.q.dtype)
        ws = torch.zeros(n, dtype=torch.uint8, device="cuda") if n else None
        _native.kda_chunk_prefill_ws(q, k, v, g, beta, case.scale, cuda(case.init_state), cu, out,
                                     fin, ws)
    else:
        _native.kda_chunk_prefill_noalloc(q, k, v, g, beta, case.scale, cuda(case.init_state), cu,
                                          out, fin)
    torch.cuda.synchronize()
    return out.cpu(), fin.cpu()


@pytest.mark.parametrize("lens,H,dtype,K", [([300, 77, 0, 130], 4, "bf16", 128),
                                            ([4096], 32, "bf16", 128),
                                            ([70, 3], 2, "f32", 128)])
def test_noalloc_equals_workspace_entry_point_twice(lens, H, dtype, K):
    case = inputs.prefill_case(lens, H=H, K=K, V=128, dtype=dtype, seed=190 + H, init_std=0.02)
    o_ref, f_ref = _run(case, "ws")
    for _ in range(2):   # the second call runs on the first call's leftovers in the scratch
        o, f = _run(case, "noalloc")
        assert torch.equal(o.view(torch.int32), o_ref.view(torch.int32))
        assert torch.equal(f.view(torch.int32), f_ref.view(torch.int32))
