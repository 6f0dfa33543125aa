"""The C-ABI library: loads, exports what include/moe.h declares, validates
arguments on the host (CPU only: no call here reaches a kernel launch)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "moe.h")


@pytest.fixture(scope="module")
def L():
    from token_dispatch_grouped_moe_gb300 import build, lib
    build.build()
    return lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(moe_[a-z_0-9]+)\s*\(", text)))


def test_exports_match_header(L):
    from token_dispatch_grouped_moe_gb300 import lib
    names = declared_functions()
    assert names, "no declarations parsed"
    for n in names:
        assert hasattr(L, n), f"{n} declared in moe.h but not exported"
    assert sorted(lib.EXPORTS) == sorted(n for n in names if n in lib.EXPORTS)
    assert set(lib.EXPORTS) <= set(names)


def test_version_and_status_strings(L):
    assert L.moe_version() >= 100
    for code in range(0, 7):
        s = L.moe_status_string(code).decode()
        assert s.startswith("MOE_")
    assert L.moe_status_string(99) == b"unknown moe_status"


def test_workspace_size(L):
    from token_dispatch_grouped_moe_gb300 import lib
    d = lib.make_dims(8192, 4096, 14336, 8, 2)
    n = lib.workspace_size(d)
    # h (R*F bf16) + slot (k*T*H f32) dominate
    assert n >= 16384 * 14336 * 2 + 2 * 8192 * 4096 * 4
    assert n % 256 == 0
    for bad in [lib.make_dims(-1, 64, 64, 8, 2), lib.make_dims(8, 60, 64, 8, 2),
                lib.make_dims(8, 64, 64, 8, 9), lib.make_dims(8, 64, 64, 300, 2),
                lib.make_dims(8, 64, 64, 2, 3)]:
        assert lib.workspace_size(bad) == 0
    assert L.moe_workspace_size(None) == 0


def test_host_validation_without_launch(L):
    """Errors found on the host return before any CUDA call."""
    from token_dispatch_grouped_moe_gb300 import lib
    dummy = ctypes.c_void_p(256)
    null = None
    # null dims
    assert L.moe_route(None, dummy, dummy, null, dummy, dummy, null) == 1
    # unsupported: H not a multiple of 64; k > 8; E > 256
    for d, want in [(lib.make_dims(8, 96, 64, 8, 2), 2), (lib.make_dims(8, 64, 64, 16, 9), 2),
                    (lib.make_dims(8, 64, 64, 300, 2), 2), (lib.make_dims(8, 64, 64, 4, 5), 1)]:
        assert L.moe_route(ctypes.byref(d), dummy, dummy, null, dummy, dummy, null) == want
    d = lib.make_dims(8, 64, 64, 8, 2)
    # missing pointers
    assert L.moe_route(ctypes.byref(d), null, dummy, null, dummy, dummy, null) == 1
    # misaligned x
    assert L.moe_route(ctypes.byref(d), ctypes.c_void_p(257), dummy, null, dummy, dummy, null) == 1
    # workspace: null, misaligned, too small
    need = lib.workspace_size(d)
    args = [ctypes.byref(d), dummy, dummy, dummy, dummy, dummy, null, null]
    assert L.moe_permute(*args, null, need, null) == 3
    assert L.moe_permute(*args, ctypes.c_void_p(4096 + 16), need, null) == 3
    assert L.moe_permute(*args, ctypes.c_void_p(4096), need - 1, null) == 3
    # combine: slot count out of range
    assert L.moe_combine(ctypes.byref(d), dummy, 0, dummy, null) == 1
    assert L.moe_combine(ctypes.byref(d), dummy, 10, dummy, null) == 1
    # shared expert weights required when F_shared > 0
    ds = lib.make_dims(8, 64, 64, 8, 2, 64)
    assert L.moe_layer_forward(ctypes.byref(ds), dummy, dummy, null, dummy, dummy, dummy, null, null,
                               null, dummy, null, ctypes.c_void_p(4096), lib.workspace_size(ds), null,
                               null) == 1


def test_host_entry_validation_without_launch(L):
    """moe_layer_forward_host rejects bad arguments before any copy or launch."""
    from token_dispatch_grouped_moe_gb300 import lib
    dummy = ctypes.c_void_p(256)
    null = None
    d = lib.make_dims(1000, 64, 64, 8, 2)
    ws, need = ctypes.c_void_p(4096), lib.workspace_size(d)

    def call(x_host=dummy, out_host=dummy, x_dev=dummy, out_dev=dummy, n_chunks=0, w=ws, nbytes=need):
        return L.moe_layer_forward_host(ctypes.byref(d), x_host, dummy, null, dummy, dummy, dummy, null, null,
                                        null, out_host, x_dev, out_dev, n_chunks, w, nbytes, null)

    assert call(x_host=null) == 1
    assert call(out_host=null) == 1
    assert call(x_dev=null) == 1
    assert call(out_dev=ctypes.c_void_p(264)) == 1   # staging buffers must be 16-byte aligned
    assert call(n_chunks=-1) == 1
    assert call(n_chunks=65) == 1
    assert call(w=null) == 3
    assert call(nbytes=need - 1) == 3
    # no tokens: nothing to do, nothing touched
    d0 = lib.make_dims(0, 64, 64, 8, 2)
    assert L.moe_layer_forward_host(ctypes.byref(d0), null, null, null, null, null, null, null, null, null,
                                    null, null, null, 0, ws, lib.workspace_size(d0), null) == 0


def test_nvtx_range_recorded(tmp_path):
    """The library's NVTX ranges reach a tool: a small NVTX tool library
    (tests/nvtx_recorder.c, loaded through NVTX_INJECTION64_PATH) records the
    pushes and pops of a child process whose host-buffer call opens its range
    and returns (no device here) with the range closed."""
    import shutil
    import subprocess
    import sys
    import torch
    if torch.cuda.is_available():
        pytest.skip("the call would run on a GPU; this test wants it to stop at the first CUDA call")
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from token_dispatch_grouped_moe_gb300 import build
    build.build()
    tool = tmp_path / "libnvtx_recorder.so"
    inc = os.path.join(os.environ.get("CUDA_HOME", "/usr/local/cuda"), "include")
    subprocess.run([cc, "-shared", "-fPIC", "-O1", "-I", inc, os.path.join(ROOT, "tests", "nvtx_recorder.c"),
                    "-o", str(tool)], check=True)
    log = tmp_path / "nvtx.log"
    child = (
        "import ctypes, sys\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from token_dispatch_grouped_moe_gb300 import lib\n"
        "L = lib.load()\n"
        "d = lib.make_dims(1000, 64, 64, 8, 2)\n"
        "p = ctypes.c_void_p(256)\n"
        "st = L.moe_layer_forward_host(ctypes.byref(d), p, p, None, p, p, p, None, None, None, p, p, p, 0,\n"
        "                              ctypes.c_void_p(4096), lib.workspace_size(d), None)\n"
        "print(st)\n")
    env = dict(os.environ, NVTX_INJECTION64_PATH=str(tool), MOE_NVTX_LOG=str(log))
    r = subprocess.run([sys.executable, "-c", child], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "4"   # MOE_ERR_CUDA: no device behind the first CUDA call
    assert log.read_text().splitlines() == ["push moe/layer_forward_host", "pop"]


def test_host_chunks_table(L):
    """The library's chunk count: >= 8192 tokens a chunk, at most three."""
    from token_dispatch_grouped_moe_gb300 import lib
    for T, want in [(1, 1), (256, 1), (8191, 1), (8192, 1), (16383, 1), (16384, 2), (32768, 3), (65536, 3)]:
        assert lib.host_chunks(lib.make_dims(T, 4096, 14336, 8, 2)) == want
    assert L.moe_host_chunks(None) == 0


def test_options(L):
    from token_dispatch_grouped_moe_gb300 import lib
    assert lib.get_gemm0_a() == lib.GEMM0_A_PERMUTED
    lib.set_gemm0_a(lib.GEMM0_A_TMA_GATHER)
    assert lib.get_gemm0_a() == lib.GEMM0_A_TMA_GATHER
    lib.set_gemm0_a(lib.GEMM0_A_PERMUTED)
    assert L.moe_set_option(0, 7) == 1
    assert L.moe_set_option(6, 0) == 1
    assert L.moe_get_option(6) == -1
    assert lib.get_combine() == lib.COMBINE_AUTO
    for mode in (lib.COMBINE_FUSED, lib.COMBINE_SEPARATE, lib.COMBINE_AUTO):
        lib.set_combine(mode)
        assert lib.get_combine() == mode
    assert L.moe_set_option(1, 3) == 1
    assert lib.get_gemm_fusion() == lib.GEMM_FUSION_AUTO
    for mode in (lib.GEMM_FUSION_ON, lib.GEMM_FUSION_OFF, lib.GEMM_FUSION_AUTO):
        lib.set_gemm_fusion(mode)
        assert lib.get_gemm_fusion() == mode
    assert L.moe_set_option(2, 3) == 1
    assert lib.get_cta_group() == lib.CTA_GROUP_AUTO
    for mode in (lib.CTA_GROUP_ONE, lib.CTA_GROUP_PAIR, lib.CTA_GROUP_AUTO):
        lib.set_cta_group(mode)
        assert lib.get_cta_group() == mode
    assert L.moe_set_option(3, 3) == 1
    assert lib.get_x_perm_copy() == lib.X_PERM_COPY_AUTO
    for mode in (lib.X_PERM_COPY_INLINE, lib.X_PERM_COPY_KERNEL, lib.X_PERM_COPY_AUTO):
        lib.set_x_perm_copy(mode)
        assert lib.get_x_perm_copy() == mode
    assert L.moe_set_option(4, 3) == 1


def test_zero_tokens_is_noop_on_host(L):
    """T = 0 returns MOE_OK before touching any pointer or the device, and
    launches nothing."""
    from token_dispatch_grouped_moe_gb300 import lib
    d = lib.make_dims(0, 64, 64, 8, 2)
    n0 = lib.launch_count()
    assert L.moe_route(ctypes.byref(d), None, None, None, None, None, None) == 0
    assert L.moe_combine(ctypes.byref(d), None, 1, None, None) == 0
    assert lib.launch_count() == n0


def test_layer_plan_table(L):
    """The per-shape table: router, combine form, GEMM fusion and CTAs per MMA
    chosen for the layer configurations (host only), and the options that
    override it."""
    from token_dispatch_grouped_moe_gb300 import lib
    from token_dispatch_grouped_moe_gb300.configs import CONFIGS
    want = {   # config: (router, combine, gemm_fusion, CTAs per MMA of GEMM0 and of GEMM1)
        "tiny": (lib.ROUTER_STREAM, lib.COMBINE_SEPARATE, lib.GEMM_FUSION_ON, 1, 1),
        "mixtral": (lib.ROUTER_STREAM, lib.COMBINE_FUSED, lib.GEMM_FUSION_OFF, 2, 2),
        "qwen2": (lib.ROUTER_TENSOR, lib.COMBINE_FUSED, lib.GEMM_FUSION_OFF, 1, 2),
        "dsk-1k": (lib.ROUTER_SLICED, lib.COMBINE_SEPARATE, lib.GEMM_FUSION_ON, 1, 1),
        "dsk-4k": (lib.ROUTER_TENSOR, lib.COMBINE_SEPARATE, lib.GEMM_FUSION_ON, 1, 1),
        "dsk-16k": (lib.ROUTER_TENSOR, lib.COMBINE_SEPARATE, lib.GEMM_FUSION_OFF, 2, 2),
        "dsk-32k": (lib.ROUTER_TENSOR, lib.COMBINE_SEPARATE, lib.GEMM_FUSION_OFF, 2, 2),
    }
    for name, (router, combine, fusion, cg, cg1) in want.items():
        c = CONFIGS[name]
        p = lib.layer_plan(lib.make_dims(c.T, c.H, c.F, c.E, c.k, c.Fs))
        assert (p.router, p.combine, p.gemm_fusion, p.cta_group, p.cta_group_gemm1) == (
            router, combine, fusion, cg, cg1), name
        tile = (256, 256, 64, 6) if cg == 2 else (128, 256, 64, 4)
        assert (p.gemm0_a, p.tile_m, p.tile_n, p.tile_k, p.stages) == (lib.GEMM0_A_PERMUTED, *tile), name
        # x_perm is filled by a copy kernel unless the option asks for the in-GEMM0 copy
        assert p.x_perm_copy == lib.X_PERM_COPY_KERNEL, name
    # the CTA-group option overrides the table; a gather A path runs one CTA
    d = lib.make_dims(8192, 4096, 14336, 8, 2)
    try:
        lib.set_cta_group(lib.CTA_GROUP_ONE)
        assert (lib.layer_plan(d).cta_group, lib.layer_plan(d).cta_group_gemm1) == (1, 1)
        lib.set_cta_group(lib.CTA_GROUP_PAIR)
        small = lib.make_dims(64, 256, 64, 8, 2)
        assert (lib.layer_plan(small).cta_group, lib.layer_plan(small).cta_group_gemm1) == (1, 1)  # one launch
        lib.set_gemm_fusion(lib.GEMM_FUSION_OFF)
        assert (lib.layer_plan(small).cta_group, lib.layer_plan(small).cta_group_gemm1) == (2, 2)
        lib.set_cta_group(lib.CTA_GROUP_AUTO)
        lib.set_x_perm_copy(lib.X_PERM_COPY_INLINE)
        assert lib.layer_plan(d).x_perm_copy == lib.X_PERM_COPY_INLINE
        lib.set_gemm_fusion(lib.GEMM_FUSION_ON)   # one launch: x_perm by the kernel
        assert lib.layer_plan(small).x_perm_copy == lib.X_PERM_COPY_KERNEL
        lib.set_gemm_fusion(lib.GEMM_FUSION_OFF)
        lib.set_x_perm_copy(lib.X_PERM_COPY_AUTO)
        lib.set_gemm0_a(lib.GEMM0_A_TMA_GATHER)
        assert (lib.layer_plan(d).cta_group, lib.layer_plan(d).cta_group_gemm1) == (1, 2)
        assert lib.layer_plan(d).x_perm_copy == 0   # GEMM0 gathers its rows: no x_perm
    finally:
        lib.set_cta_group(lib.CTA_GROUP_AUTO)
        lib.set_x_perm_copy(lib.X_PERM_COPY_AUTO)
        lib.set_gemm_fusion(lib.GEMM_FUSION_AUTO)
        lib.set_gemm0_a(lib.GEMM0_A_PERMUTED)
    # E not a multiple of 8, E > 64, a gate too large for the streaming router
    assert lib.layer_plan(lib.make_dims(64, 256, 64, 12, 2)).router == lib.ROUTER_CLUSTER
    assert lib.layer_plan(lib.make_dims(64, 256, 64, 200, 2)).router == lib.ROUTER_SLICED
    assert lib.layer_plan(lib.make_dims(64, 256, 64, 196, 2)).router == lib.ROUTER_BLOCK
    assert lib.layer_plan(lib.make_dims(64, 16384, 64, 8, 2)).router == lib.ROUTER_BLOCK
    # the tensor-core router by default for 16 <= E <= 64 (a multiple of 8)
    # from 4096 tokens; forced by the option from 512 tokens and E >= 8; the
    # other option value keeps the FMA routers
    assert lib.layer_plan(lib.make_dims(4096, 256, 64, 64, 6)).router == lib.ROUTER_TENSOR
    assert lib.layer_plan(lib.make_dims(4095, 256, 64, 64, 6)).router == lib.ROUTER_SLICED
    assert lib.layer_plan(lib.make_dims(65536, 4096, 64, 8, 2)).router == lib.ROUTER_STREAM
    assert lib.layer_plan(lib.make_dims(16384, 256, 64, 12, 2)).router == lib.ROUTER_CLUSTER
    assert lib.layer_plan(lib.make_dims(16384, 256, 64, 72, 2)).router == lib.ROUTER_SLICED
    try:
        lib.set_router(lib.ROUTER_OPT_TENSOR)
        assert lib.layer_plan(lib.make_dims(512, 256, 64, 64, 6)).router == lib.ROUTER_TENSOR
        assert lib.layer_plan(lib.make_dims(8192, 4096, 64, 8, 2)).router == lib.ROUTER_TENSOR
        assert lib.layer_plan(lib.make_dims(511, 256, 64, 64, 6)).router == lib.ROUTER_SLICED
        lib.set_router(lib.ROUTER_OPT_FMA)
        assert lib.layer_plan(lib.make_dims(32768, 2048, 64, 64, 6)).router == lib.ROUTER_SLICED
    finally:
        lib.set_router(lib.ROUTER_OPT_AUTO)
    # options override the automatic entries; a gather A path rules out fusion
    d = lib.make_dims(1024, 2048, 1408, 64, 6)
    try:
        lib.set_combine(lib.COMBINE_FUSED)
        lib.set_gemm_fusion(lib.GEMM_FUSION_OFF)
        p = lib.layer_plan(d)
        assert (p.combine, p.gemm_fusion) == (lib.COMBINE_FUSED, lib.GEMM_FUSION_OFF)
        lib.set_gemm_fusion(lib.GEMM_FUSION_ON)
        lib.set_gemm0_a(lib.GEMM0_A_TMA_GATHER)
        assert lib.layer_plan(d).gemm_fusion == lib.GEMM_FUSION_OFF
    finally:
        lib.set_combine(lib.COMBINE_AUTO)
        lib.set_gemm_fusion(lib.GEMM_FUSION_AUTO)
        lib.set_gemm0_a(lib.GEMM0_A_PERMUTED)
    with pytest.raises(lib.MoeError):
        lib.layer_plan(lib.make_dims(64, 100, 64, 8, 2))   # H not a multiple of 64


def test_c_example_compiles(L, tmp_path):
    """include/example.c (one layer call in C) compiles and links against
    include/moe.h and the library (no GPU: it is not run)."""
    import shutil
    import subprocess
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    src = os.path.join(root, "include", "example.c")
    cuda = os.environ.get("CUDA_HOME", "/usr/local/cuda")
    gcc = shutil.which("gcc")
    if gcc is None or not os.path.exists(os.path.join(cuda, "include", "cuda_runtime.h")):
        pytest.skip("no C compiler or CUDA headers")
    pkg = os.path.join(root, "token_dispatch_grouped_moe_gb300")
    cmd = [gcc, "-std=c11", "-Wall", "-Werror", "-DMOE_EXAMPLE_MAIN", "-I", os.path.join(root, "include"),
           "-I", os.path.join(cuda, "include"), src, "-o", str(tmp_path / "example"), "-L", pkg,
           "-lmoe_gb300", "-L", os.path.join(cuda, "lib64"), "-lcudart"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr

