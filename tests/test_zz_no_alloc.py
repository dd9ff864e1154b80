"""spec_linear_noalloc: the projection entry point for callers that cannot
allocate device memory (a host that owns the whole device-memory budget, a
plugin whose framework allocator must see every allocation, or code that must
not reach cudaMalloc because it may synchronise the device). Its scratch is a
fixed array inside the library that every call reuses, so the test checks two
calls in a row: each against the oracle's exact fp64 linear layer at the
kernel-level tolerance, and against spec_linear on the same inputs. Row counts
above 8 run there as 8-row passes sharing that one array, so M = 9, 40 and 64
are covered too. Collected last so that a failure here comes after every other
test has run."""
import ctypes as C

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_spec_gb300 import binding, configs, synth
from tests.parity import assert_rows_close

pytestmark = pytest.mark.gpu

TOL = 1e-4  # the kernel-level tolerance of the projection tests


def _x(M, K, seed):
    return torch.randn((M, K), generator=torch.Generator(device="cuda").manual_seed(seed), device="cuda")


def _rms_gain(x, gain, eps=1e-6):
    """The input the kernel projects, through the oracle's RMSNorm when a gain
    is given."""
    xd = x.double().cpu().numpy()
    if gain is None:
        return xd
    g = gain.cpu().numpy()
    return np.stack([oracle.rmsnorm(row, g, eps) for row in xd])


@pytest.mark.parametrize("dtype,N,K,M,norm", [
    (configs.BF16, 4112, 1536, 5, False),      # ragged N
    (configs.BF16, 1536, 6144, 4, True),       # long K, fused RMSNorm
    (configs.Q4_0, 1000, 1536, 3, True),
    (configs.BF16, 1000, 1536, 9, False),      # 8-row passes: 8 + 1
    (configs.BF16, 4112, 2048, 40, True),
    (configs.BF16, 300, 256, 64, False),
    (configs.Q4_0, 1000, 1536, 9, False),
    (configs.Q4_0, 4112, 2048, 40, True),
    (configs.Q4_0, 300, 256, 64, False),
])
def test_noalloc_matches_oracle_and_spec_linear_on_two_calls(dtype, N, K, M, norm):
    from speculative_decoding_spec_gb300 import build
    build.build()
    g = torch.Generator(device="cuda").manual_seed(N + K)
    w = synth.make_matrix(g, dtype, 1, N, K, 0.02, "cuda")
    gain = (torch.rand(K, generator=g, device="cuda") + 0.5) if norm else None
    for call in range(2):
        x = _x(M, K, 1 + call)
        y = binding.spec_linear_noalloc(w, x, gain=gain)
        ref = binding.spec_linear(w, x, gain=gain)
        torch.cuda.synchronize()
        exact = oracle.linear(w, _rms_gain(x, gain))
        assert_rows_close(y.cpu().numpy(), exact, TOL, "noalloc call %d vs oracle" % call)
        assert_rows_close(y.cpu().numpy(), ref.cpu().numpy(), TOL, "noalloc call %d vs spec_linear" % call)


def test_noalloc_rejects_oversized_n():
    L = binding.lib()
    N = binding.SPEC_LINEAR_NOALLOC_MAX_ROWS + 1
    w = synth.make_matrix(torch.Generator(device="cuda").manual_seed(0), configs.BF16, 1, 16, 256, 0.02, "cuda")
    m = binding.spec_matrix(1, w.data.data_ptr(), None)
    x = _x(1, 256, 0)
    y = torch.empty((1, 16), device="cuda")
    rc = L.spec_linear_noalloc(C.byref(m), N, 256, x.data_ptr(), 1, None, 0.0, y.data_ptr(), None)
    assert rc == binding.SPEC_ECAPACITY
