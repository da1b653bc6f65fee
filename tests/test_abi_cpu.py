"""CPU-only checks of the boundary: the library builds for sm_103a, loads
without a GPU, exports every symbol include/flce.h declares, agrees with the
binding on the options layout, and plans workspaces as documented."""
import os
import re
import shutil
import subprocess

import pytest

import linear_cross_entropy_fwd_gb300 as flce
from linear_cross_entropy_fwd_gb300 import build as flce_build
from flce_synth import WORKLOADS

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    flce_build.build()
    return flce.load_library()


def _declared():
    src = open(os.path.join(ROOT, "include", "flce.h")).read()
    return re.findall(r"FLCE_API\s+[\w\s\*]+?\b(flce_\w+)\s*\(", src)


def test_header_declares_the_boundary():
    names = _declared()
    for must in ["flce_fwd_bwd", "flce_fwd_bwd_ex", "flce_fwd", "flce_fwd_bwd_host",
                 "flce_workspace_bytes", "flce_status_str", "flce_last_error",
                 "flce_opts_init"]:
        assert must in names
    assert sorted(names) == sorted(flce.EXPORTED)


def test_library_exports_every_declared_symbol(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_opts_layout_and_version(lib):
    import ctypes
    assert lib.flce_opts_sizeof() == ctypes.sizeof(flce.FlceOpts)
    assert lib.flce_version() == 2
    o = flce.make_opts()
    assert o.sync == 1 and o.grad_scale == 1.0 and o.dtype == flce.FLCE_BF16


def test_status_strings(lib):
    for s in range(8):
        assert lib.flce_status_str(s)
    assert lib.flce_status_str(999) == b"unknown status"


def test_workspace_plans(lib):
    # loss only: no gradient chunk, no dX accumulator
    w = WORKLOADS["llama3_8b_head_8192x4096x128256"]
    fwd = flce.flce_workspace_bytes(w.N, w.H, w.V, with_grads=False)
    assert fwd < 20 * 2 ** 20
    for name in ["llama3_8b_head_8192x4096x128256", "long_context_65536x4096x128256",
                 "qwen2_7b_head_16384x3584x152064"]:
        w = WORKLOADS[name]
        ws = flce.flce_workspace_bytes(w.N, w.H, w.V)
        assert 0 < ws <= w.N * w.V * 4 // 16, name
    # an explicit chunk width is honoured; a smaller budget gives a smaller plan
    a = flce.flce_workspace_bytes(8192, 4096, 128256, vocab_chunk=1024)
    b = flce.flce_workspace_bytes(8192, 4096, 128256, vocab_chunk=2048)
    assert b - a == 8192 * 1024 * 2
    # a budget below what a 2048-column chunk needs gets the 2048-column plan
    small = flce.flce_workspace_bytes(8192, 4096, 128256, workspace_budget=150 * 2 ** 20)
    assert small == flce.flce_workspace_bytes(8192, 4096, 128256, vocab_chunk=2048)
    mid = flce.flce_workspace_bytes(8192, 4096, 128256, workspace_budget=200 * 2 ** 20)
    assert small < mid <= 200 * 2 ** 20
    # bad sizes plan nothing
    assert flce.flce_workspace_bytes(10, 0, 5) == 0
    assert flce.flce_workspace_bytes(10, 8, 5, vocab_chunk=300) == 0


@pytest.mark.parametrize("name,vc", [
    ("small_head_2048x2048x32000", 20224),        # 96 MiB budget floor: 2 chunks
    ("llama3_8b_head_8192x4096x128256", 4864),    # pass 2 / dW fill 8 / 4 whole waves
    ("qwen2_7b_head_16384x3584x152064", 9728),
    ("long_context_65536x4096x128256", 4864),
])
def test_default_chunk_widths(lib, name, vc):
    """The planner's default chunk width for each workload, read back from the
    workspace size (the G chunk is N x Vc bf16 on top of a fixed part)."""
    w = WORKLOADS[name]
    base = flce.flce_workspace_bytes(w.N, w.H, w.V, vocab_chunk=256)
    ws = flce.flce_workspace_bytes(w.N, w.H, w.V)
    assert (ws - base) % (w.N * 2) == 0
    assert 256 + (ws - base) // (w.N * 2) == vc


def test_product_path_has_no_oracle_import():
    """The CUDA package never reaches into the oracle or the generator."""
    pkg = os.path.join(ROOT, "linear_cross_entropy_fwd_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "oracle" not in src.replace("oracle/", ""), f
                assert "flce_synth" not in src, f


@pytest.mark.parametrize("std,lang", [("c99", "c"), ("c++11", "c++")])
def test_header_is_plain_c(tmp_path, std, lang):
    """include/flce.h needs no CUDA or C++ header: a C99 program (and a C++11
    one) that fills the options and names every entry point compiles."""
    cc = shutil.which("gcc" if lang == "c" else "g++")
    if cc is None:
        pytest.skip("no host compiler")
    calls = "\n".join(f"  (void)&{n};" for n in _declared())
    src = tmp_path / ("h.c" if lang == "c" else "h.cpp")
    src.write_text('#include "flce.h"\nint main(void) {\n  flce_opts o;\n'
                   '  flce_opts_init(&o);\n' + calls + "\n  return 0;\n}\n")
    r = subprocess.run([cc, f"-std={std}", "-Wall", "-Wextra", "-Werror", "-fsyntax-only",
                        "-I", os.path.join(ROOT, "include"), str(src)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_tile_orders_cover_every_tile_once(tmp_path):
    """The GEMM launches' tile orders (M fastest, N fastest, M fastest in
    bands of M blocks, N fastest in bands of N blocks, ragged last band) map
    the tile indices one to one onto the tile grid: the engine's own
    tile_coords, compiled for the host."""
    cxx = shutil.which("g++")
    if cxx is None:
        pytest.skip("no host compiler")
    src = tmp_path / "tiles.cpp"
    src.write_text(r'''
#include <cstdio>
#include <vector>
#define __host__
#define __device__
#include "flce_internal.h"
int main() {
  int bad = 0;
  for (int nm : {1, 2, 5, 16, 17, 32, 64, 256})
    for (int nn : {1, 3, 19, 501, 594})
      for (int raster : {0, 1})
        for (int band : {0, 1, 3, 8, 16, 18, 40}) {
          flce::GemmGrid g{};
          g.num_m_blk = nm; g.num_n_blk = nn; g.raster_n = raster;
          (raster ? g.n_band : g.m_band) = band;
          std::vector<int> seen(nm * nn, 0);
          for (int t = 0; t < nm * nn; ++t) {
            int m, n;
            flce::tile_coords(g, t, m, n);
            if (m < 0 || m >= nm || n < 0 || n >= nn) { ++bad; continue; }
            ++seen[m * nn + n];
          }
          for (int v : seen) bad += (v != 1);
        }
  std::printf("%d\n", bad);
  return bad != 0;
}
''')
    exe = tmp_path / "tiles"
    csrc = os.path.join(ROOT, "linear_cross_entropy_fwd_gb300", "csrc")
    r = subprocess.run([cxx, "-std=c++17", "-I", csrc, str(src), "-o", str(exe)],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([str(exe)], capture_output=True, text=True)
    assert r.returncode == 0 and r.stdout.strip() == "0", r.stdout


def test_binding_checks_output_buffers():
    """The binding refuses an output buffer of the wrong shape, dtype or
    layout before anything reaches the library (no device needed)."""
    import torch
    ok = torch.empty(5, dtype=torch.float32)
    flce._check_out(ok, (5,), torch.float32, ok.device, "lse_out")
    for bad in (torch.empty(4, dtype=torch.float32), torch.empty(5, dtype=torch.float64),
                torch.empty(10, dtype=torch.float32)[::2]):
        with pytest.raises(ValueError):
            flce._check_out(bad, (5,), torch.float32, ok.device, "lse_out")
    with pytest.raises(ValueError):
        flce._check_row_outs(5, ok.device, torch.empty(6), None)
    assert flce._is32(torch.zeros(3, dtype=torch.int32)) == 1
    assert flce._is32(torch.zeros(3, dtype=torch.int64)) == 0
