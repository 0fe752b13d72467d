"""The C ABI library loads on a CPU-only machine and exports every declared function."""
import ctypes
import os

import pytest

from fac_whitening_gb300 import gift as G


def _lib_or_skip():
    try:
        return G.lib()
    except RuntimeError as e:  # not built in this checkout
        pytest.skip(str(e))


def test_exports_every_declared_function():
    lib = _lib_or_skip()
    names = G.header_functions()
    assert len(names) >= 12
    for name in names:
        assert hasattr(lib, name), name


def test_host_only_helpers():
    _lib_or_skip()
    assert G.gift_version() == 1
    assert G.status_string(G.OK) == "ok"
    assert G.status_string(G.ERR_NOT_PD).startswith("factor")
    assert G.gift_code_sizes("e4m3", "tensor", 10, 20) == (200, 1)
    assert G.gift_code_sizes("e5m2", "block128", 300, 200) == (60000, 6)
    assert G.gift_code_sizes("nvfp4", "tensor", 4, 32) == (64, 8)
    assert G.gift_code_sizes("f32", "tensor", 3, 5) == (60, 0)
    with pytest.raises(G.GiftError):
        G.gift_code_sizes("nvfp4", "tensor", 4, 30)   # d_in not a multiple of 16
    with pytest.raises(G.GiftError):
        G.gift_code_sizes("e4m3", "tensor", 0, 5)


def test_null_context_is_rejected():
    lib = _lib_or_skip()
    assert lib.gift_create(None, 0) == G.ERR_INVALID_ARG
    assert lib.gift_set_option(None, 0, 10) == G.ERR_INVALID_ARG
    assert lib.gift_workspace_bytes(None, 1, 0, 1, 0, 4, 4, 0, 0) == ctypes.c_size_t(-1).value
    # the replica entry points check their context before anything else (no CUDA call)
    assert lib.gift_encode_replicas(None, None, 1, None, 4, 4, 1, 0, 0, None, None, None, None, None, None, 0,
                                    None, None) == G.ERR_INVALID_ARG
    assert lib.gift_encode_replicas_shared(None, None, 1, None, 4, 4, 1, 0, 0, None, None, None, None, None, 0,
                                           None, None) == G.ERR_INVALID_ARG
    assert lib.gift_amax_replicas(None, None, 1, None, 4, 4, 1, 0, 0, None, None, 0, None, None) == G.ERR_INVALID_ARG
    assert lib.gift_replica_reduce(None, 1, None, None, None, 1, 0, 4, 4, None, None, None) == G.ERR_INVALID_ARG


def test_binding_refuses_host_and_strided_buffers():
    # the binding hands the library device addresses of dense buffers only
    import torch

    assert G._p(None) is None and G._p(1234) == 1234
    with pytest.raises(ValueError, match="device memory"):
        G._p(torch.zeros(4))

    class StridedCuda:   # stands in for a CUDA tensor view (no GPU here)
        is_cuda = True

        def is_contiguous(self):
            return False

        def data_ptr(self):
            return 4096

    class DenseCuda(StridedCuda):
        def is_contiguous(self):
            return True

    with pytest.raises(ValueError, match="contiguous"):
        G._p(StridedCuda())
    assert G._p(DenseCuda()) == 4096


def _header_param_counts():
    import re
    text = open(G.HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    counts = {}
    for m in re.finditer(r"(gift_[a-z0-9_]+)\s*\(([^;{]*?)\)\s*;", text, re.S):
        params = m.group(2).strip()
        counts[m.group(1)] = 0 if params in ("", "void") else params.count(",") + 1
    return counts


def test_binding_declares_every_function_with_the_header_arity():
    # every declared function has a ctypes signature, with as many arguments as the header's
    lib = _lib_or_skip()
    counts = _header_param_counts()
    assert set(counts) == set(G.header_functions())
    for name, n in counts.items():
        fn = getattr(lib, name)
        assert fn.argtypes is not None, f"{name}: no ctypes signature"
        assert len(fn.argtypes) == n, f"{name}: {len(fn.argtypes)} ctypes arguments, header has {n}"


def test_c_program_links_and_calls_host_entry_points(tmp_path):
    # the boundary is a C ABI: a C99 program includes gift.h, links libgift.so and calls the
    # host-only entry points (no device needed)
    import shutil
    import subprocess
    _lib_or_skip()
    cuda_inc = "/usr/local/cuda/include"
    if shutil.which("gcc") is None or not os.path.isdir(cuda_inc):
        pytest.skip("gcc or the CUDA headers are not available")
    src = tmp_path / "consumer.c"
    src.write_text(r"""
#include <stdio.h>
#include "gift.h"
int main(void) {
  size_t cb = 0, sc = 0;
  unsigned long long counts[6] = {1, 9, 100, 0, 1, 100};
  int order[2] = {-1, -1}, k = -1;
  double scores[2];
  if (gift_code_sizes(GIFT_FMT_NVFP4, GIFT_SCALE_TENSOR, 4, 32, &cb, &sc) != GIFT_OK) return 2;
  if (gift_select_fragile(2, counts, 1, 1, 2, order, scores, &k) != GIFT_OK) return 3;
  printf("%d %zu %zu %d %d %d %s\n", gift_version(), cb, sc, order[0], order[1], k,
         gift_status_string(GIFT_ERR_INVALID_ARG));
  return 0;
}
""")
    exe = tmp_path / "consumer"
    libdir = os.path.dirname(G.LIB_PATH)
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", f"-I{os.path.dirname(G.HEADER)}", f"-I{cuda_inc}",
                    str(src), "-o", str(exe), f"-L{libdir}", "-lgift", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert out[:6] == ["1", "64", "8", "0", "1", "1"]
    assert " ".join(out[6:]) == G.status_string(G.ERR_INVALID_ARG)
