"""The C ABI library loads without a GPU, exports every entry point that
include/spec.h declares, and rejects invalid calls on the host before any
launch."""
import ctypes as C
import os
import re

import pytest

from speculative_decoding_spec_gb300 import binding, configs

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
            names |= set(re.findall(r"\b(spec_[a-z0-9_]+)\s*\(", src))
    return names


@pytest.fixture(scope="module")
def lib():
    from speculative_decoding_spec_gb300 import build
    build.build()
    return binding.lib()


def test_every_declared_entry_point_is_exported(lib):
    declared = _declared()
    assert declared, "no declarations found"
    for name in sorted(declared):
        assert hasattr(lib, name), name
    assert set(binding.EXPORTS) <= declared


def test_status_strings(lib):
    assert lib.spec_status_str(0) == b"ok"
    assert lib.spec_status_str(2) == b"capacity exceeded"


def test_invalid_descriptors_rejected_on_host(lib):
    md = binding.model_desc(configs.E2B)
    assert lib.spec_workspace_bytes(C.byref(md), None, 1, 4, 33) > 0
    bad = binding.model_desc(configs.E2B)
    bad.n_kv_heads = 5                      # 12 query heads do not group onto 5
    assert lib.spec_workspace_bytes(C.byref(bad), None, 1, 4, 33) == 0
    assert lib.spec_workspace_bytes(C.byref(md), None, 0, 4, 33) == 0
    ctx = C.c_void_p()
    assert lib.spec_init(None, None, None, None, None, None, 1, 4, None, 0, None,
                         C.byref(ctx)) == binding.SPEC_EINVAL
    # calls on a null context are rejected without touching the device
    assert lib.spec_verify(None, 1, None, 3, None, None, None, None, None) == binding.SPEC_EINVAL
    assert lib.spec_sync(None, None) == binding.SPEC_EINVAL


def test_workspace_scales_with_batch_and_rows(lib):
    md = binding.model_desc(configs.E4B)
    dd = binding.drafter_desc(configs.WORKLOADS["e4b_bf16_b8_ragged_k4"].drafter)
    a = lib.spec_workspace_bytes(C.byref(md), C.byref(dd), 1, 5, 129)
    b = lib.spec_workspace_bytes(C.byref(md), C.byref(dd), 8, 5, 129)
    assert b > a > 0
