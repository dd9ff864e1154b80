"""spec_linear_noalloc: the projection entry point for callers that cannot
allocate device memory (its scratch is a fixed array inside the library).
Its results must equal spec_linear's, call after call, since every call reuses
the same scratch. Collected last so a failure here comes after every other
test has run."""
import ctypes as C

import pytest
import torch

from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import assert_rows_close

pytestmark = pytest.mark.gpu

TOL = 1e-4  # the kernel-level tolerance of the projection tests


def _x(M, K, seed):
    return torch.randn((M, K), generator=torch.Generator(device="cuda").manual_seed(seed), device="cuda")


@pytest.mark.parametrize("dtype,N,K,M,norm", [
    (configs.BF16, 4112, 1536, 5, False),      # ragged N, tensor-core path with split tiles
    (configs.BF16, 1536, 6144, 4, True),       # long K, fused RMSNorm
    (configs.Q4_0, 1000, 1536, 3, True),
])
def test_noalloc_matches_spec_linear_on_two_calls(dtype, N, K, M, norm):
    from speculative_decoding_spec_gb300 import build
    build.build()
    g = torch.Generator(device="cuda").manual_seed(N + K)
    w = synth.make_matrix(g, dtype, 1, N, K, 0.02, "cuda")
    gain = (torch.rand(K, generator=g, device="cuda") + 0.5) if norm else None
    ref = binding.spec_linear(w, _x(M, K, 1), gain=gain)
    for call in range(2):
        x = _x(M, K, 1 + call)
        ref = binding.spec_linear(w, x, gain=gain)
        y = binding.spec_linear_noalloc(w, x, gain=gain)
        torch.cuda.synchronize()
        assert_rows_close(y.cpu().numpy(), ref.cpu().numpy(), TOL, "noalloc call %d" % call)


def test_noalloc_rejects_oversized_n():
    L = binding.lib()
    N = binding.SPEC_LINEAR_NOALLOC_MAX_ROWS + 1
    w = synth.make_matrix(torch.Generator(device="cuda").manual_seed(0), configs.BF16, 1, 16, 256, 0.02, "cuda")
    m = binding.spec_matrix(1, w.data.data_ptr(), None)
    x = _x(1, 256, 0)
    y = torch.empty((1, 16), device="cuda")
    rc = L.spec_linear_noalloc(C.byref(m), N, 256, x.data_ptr(), 1, None, 0.0, y.data_ptr(), None)
    assert rc == binding.SPEC_ECAPACITY
