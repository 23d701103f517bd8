"""The C ABI library loads, exports every declared symbol, and rejects bad
arguments on the host (no device work is started by any call here)."""

import ctypes
import os
import re

import pytest

import gemv_tiled_gemm_gb300 as gtg
from gemv_tiled_gemm_gb300 import _build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gtg.h")
TESTING_HEADER = os.path.join(ROOT, "include", "gtg_testing.h")


def _has_device():
    import torch
    return torch.cuda.is_available()


# Calls below that pass validation with fake addresses would launch kernels on
# a machine with a GPU; those parts run only where no device exists (there
# the call stops at the device lookup). The GPU tests cover the same paths
# with real buffers.
no_device_only = pytest.mark.skipif(_has_device(), reason="would launch with fake device addresses")


@pytest.fixture(scope="module", autouse=True)
def built():
    _build.build()
    gtg.lib()


def _declared(path):
    text = open(path).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return re.findall(r"GTG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)


def declared_functions():
    """Every exported function: the product ABI plus the testing header."""
    return _declared(HEADER) + _declared(TESTING_HEADER)


def test_header_declares_the_entry_points():
    names = set(declared_functions())
    for want in ("gemm_f32", "gemm_tf32", "gemm_bf16", "gemv_f32", "gtg_status_string",
                 "gtg_sync_status"):
        assert want in names


def test_library_exports_every_declared_symbol():
    handle = ctypes.CDLL(gtg.LIB_PATH)
    for name in declared_functions():
        assert hasattr(handle, name), f"{name} declared in gtg.h but not exported"
    # and the binding covers each one with a signature, in the matching table
    assert set(_declared(HEADER)) == set(gtg.SIGNATURES)
    assert set(_declared(TESTING_HEADER)) == set(gtg.TESTING_SIGNATURES)


def test_product_header_holds_no_testing_hook():
    names = set(_declared(HEADER))
    hooks = {n for n in names if n.startswith(("gtg_test_", "gtg_force_")) or n.endswith("_force_path")
             or n == "gtg_set_wait_limit_ns"}
    assert not hooks, hooks
    assert not set(_declared(HEADER)) & set(_declared(TESTING_HEADER))


def test_failure_hooks_need_the_testing_switch():
    # the hooks read GTG_TESTING when called; without it they arm nothing
    import subprocess
    import sys
    code = ("import gemv_tiled_gemm_gb300 as g; "
            "print(g.gtg_test_drop_load(1), g.gtg_test_skip_vector_copy(1), g.gtg_test_inject_launch_failure(1))")
    env = {k: v for k, v in os.environ.items() if k != "GTG_TESTING"}
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == [str(gtg.GTG_ERR_UNSUPPORTED)] * 3
    # with it, they arm (and are cancelled again here)
    assert gtg.gtg_test_drop_load(-1) == gtg.GTG_OK
    assert gtg.gtg_test_skip_vector_copy(False) == gtg.GTG_OK
    assert gtg.gtg_test_inject_launch_failure(0) == gtg.GTG_OK


@no_device_only
def test_injected_launch_failure_stops_the_dispatcher():
    # Valid arguments at fake addresses: without a GPU the call would fail
    # looking for the device (GTG_ERR_DEVICE); the injected failure comes
    # first, in the dispatcher, before any CUDA call. Calls that fail
    # validation do not count towards the injection.
    ok_args = (4, 4, 4, A, 4, B, 4, C, 4)
    assert gtg.gtg_test_inject_launch_failure(2) == gtg.GTG_OK
    assert gtg.gemm_f32(-1, 4, 4, A, 4, B, 4, C, 4) == gtg.GTG_ERR_INVALID_VALUE   # not counted
    first = gtg.gemm_f32(*ok_args)                                                 # counted: 1
    assert first != gtg.GTG_ERR_LAUNCH
    assert gtg.gemv_f32(4, 4, A, 4, B, 4, C, 4, 1) == gtg.GTG_ERR_LAUNCH             # counted: 2, fires
    assert gtg.last_cuda_error() == "injected launch failure"
    assert gtg.gemm_f32(*ok_args) == first                                         # disarmed again
    # every dispatching entry point takes part
    for call in (lambda: gtg.gemm_tf32(*ok_args), lambda: gtg.gemm_bf16(*ok_args),
                 lambda: gtg.gemm_tf32_noalloc(*ok_args),
                 lambda: gtg.gemm_strided_batched("bf16", 4, 4, 4, A, 4, 16, B, 4, 16, C, 4, 16, 2),
                 lambda: gtg.gemv_bf16(4, 4, A, 4, B, 4, C, 4, 2),
                 lambda: gtg.conv2d_nhwc("bf16", 1, 4, 4, 8, 8, 3, 3, 1, 1, 1, 1, 1, 1, A, B, C),
                 lambda: gtg.gemm_host("f32", 4, 4, 4, A, 4, B, 4, C, 4)):
        assert gtg.gtg_test_inject_launch_failure(1) == gtg.GTG_OK
        assert call() == gtg.GTG_ERR_LAUNCH
    assert gtg.gtg_test_inject_launch_failure(0) == gtg.GTG_OK


@no_device_only
def test_fault_inject_environment_variable():
    import subprocess
    import sys
    code = ("import gemv_tiled_gemm_gb300 as g; A, B, C = 1 << 32, 2 << 32, 3 << 32; "
            "print(*[g.gemm_f32(4, 4, 4, A, 4, B, 4, C, 4) for _ in range(4)])")
    env = {k: v for k, v in os.environ.items() if k != "GTG_TESTING"}
    env["GTG_FAULT_INJECT"] = "3"
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    st = [int(v) for v in out.stdout.split()]
    assert st[2] == gtg.GTG_ERR_LAUNCH and gtg.GTG_ERR_LAUNCH not in (st[0], st[1], st[3]), st


def test_debug_build_compiles_and_reports_itself():
    """The GTG_DEBUG variant (bounds-checking kernels) builds with the same
    sources and exports the same symbols; each library reports which it is."""
    import subprocess
    import sys
    path = _build.build(debug=True)
    assert os.path.basename(path) == "libgtg_debug.so"
    code = "import gemv_tiled_gemm_gb300 as g; print(g.gtg_debug_build(), g.gtg_test_debug_shrink_extent(0))"
    env = dict(os.environ, GTG_DEBUG="1", GTG_TESTING="1")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert out.returncode == 0, out.stderr
    assert out.stdout.split() == ["1", str(gtg.GTG_OK)]
    assert gtg.gtg_debug_build() == 0
    assert gtg.gtg_test_debug_shrink_extent(1) == gtg.GTG_ERR_UNSUPPORTED   # release build
    nm = lambda p: {l.split()[-1] for l in subprocess.run(["nm", "-D", "--defined-only", p], capture_output=True,
                                                           text=True).stdout.splitlines() if " T " in l}
    assert nm(path) == nm(gtg.LIB_PATH)


def test_only_the_c_abi_is_exported():
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", gtg.LIB_PATH], capture_output=True,
                         text=True).stdout
    text_syms = {l.split()[-1] for l in out.splitlines() if " T " in l}
    assert text_syms == set(declared_functions())


def test_status_strings():
    for s in range(8):
        assert gtg.status_string(s)
    assert "unknown" in gtg.status_string(99)


# Fake but aligned, non-overlapping "device" addresses: validation never
# dereferences them, and every call below fails validation before any CUDA call.
A, B, C = 1 << 32, 2 << 32, 3 << 32


@pytest.mark.parametrize("fn", [gtg.gemm_f32, gtg.gemm_tf32, gtg.gemm_bf16])
def test_gemm_argument_validation(fn):
    E = gtg.GTG_ERR_INVALID_VALUE
    assert fn(-1, 4, 4, A, 4, B, 4, C, 4) == E
    assert fn(4, -1, 4, A, 4, B, 4, C, 4) == E
    assert fn(4, 4, -1, A, 4, B, 4, C, 4) == E
    assert fn(4, 4, 8, A, 7, B, 4, C, 4) == E          # lda < K
    assert fn(4, 8, 4, A, 4, B, 7, C, 8) == E          # ldb < N
    assert fn(4, 8, 4, A, 4, B, 8, C, 7) == E          # ldc < N
    assert fn(4, 4, 4, A, 4, B, 4, 0, 4) == E          # null C
    assert fn(4, 4, 4, 0, 4, B, 4, C, 4) == E          # null A with K > 0
    assert fn(1 << 31, 4, 4, A, 4, B, 4, C, 4) == E    # beyond 32-bit sizes
    # empty outputs are valid and launch nothing (no device needed)
    assert fn(0, 4, 4, 0, 4, 0, 4, 0, 4) == gtg.GTG_OK
    assert fn(4, 0, 4, 0, 4, 0, 1, 0, 1) == gtg.GTG_OK


@pytest.mark.parametrize("fn,elem", [(gtg.gemm_f32, 4), (gtg.gemm_tf32, 4), (gtg.gemm_bf16, 2)])
def test_gemm_alignment_and_alias(fn, elem):
    assert fn(4, 4, 4, A + 1, 4, B, 4, C, 4) == gtg.GTG_ERR_MISALIGNED
    assert fn(4, 4, 4, A, 4, B, 4, C + 2, 4) == gtg.GTG_ERR_MISALIGNED
    # C overlapping A or B
    assert fn(4, 4, 4, A, 4, B, 4, A + 4 * elem, 4) == gtg.GTG_ERR_ALIAS
    assert fn(4, 4, 4, A, 4, B, 4, B, 4) == gtg.GTG_ERR_ALIAS
    # adjacent, touching but not overlapping, is fine as far as validation goes
    # (it then needs a device: checked only where none exists, see no_device_only)
    if not _has_device():
        st = fn(4, 4, 4, A, 4, A + 16 * elem, 4, A + 32 * elem, 4)
        assert st not in (gtg.GTG_ERR_ALIAS, gtg.GTG_ERR_INVALID_VALUE, gtg.GTG_ERR_MISALIGNED)


def test_gemm_host_argument_validation():
    E = gtg.GTG_ERR_INVALID_VALUE
    f = gtg.gemm_host
    assert f(9, 4, 4, 4, A, 4, B, 4, C, 4) == E           # no such precision
    assert f("bf16", 4, 4, 8, A, 7, B, 4, C, 4) == E      # lda < K
    assert f("f32", 4, 8, 4, A, 4, B, 8, C, 7) == E       # ldc < N
    assert f("f32", 4, 4, 4, A, 4, B, 4, 0, 4) == E       # null C
    assert f("tf32", 4, 4, 4, A, 4, B, 4, A + 16, 4) == gtg.GTG_ERR_ALIAS
    assert f("f16", 4, 4, 4, A + 1, 4, B, 4, C, 4) == gtg.GTG_ERR_MISALIGNED
    assert f("f32", 4, 4, 4, A, 4, B, 4, C, 4, gtg.epilogue(0, 7)) == E
    assert f("bf16", 0, 4, 4, 0, 4, 0, 4, 0, 4) == gtg.GTG_OK


def test_gemv_argument_validation():
    E = gtg.GTG_ERR_INVALID_VALUE
    f = gtg.gemv_f32
    assert f(-1, 4, A, 4, B, 4, C, 4, 1) == E
    assert f(4, 8, A, 7, B, 8, C, 4, 1) == E        # lda < N
    assert f(4, 4, A, 4, B, 4, C, 4, 0) == E        # batch < 1
    assert f(4, 4, A, 4, B, 4, C, 4, 9) == E        # batch > 8
    assert f(4, 8, A, 8, B, 7, C, 4, 2) == E        # ldx < N with batch > 1
    assert f(8, 4, A, 4, B, 4, C, 7, 2) == E        # ldy < M with batch > 1
    assert f(4, 4, A, 4, B, 4, 0, 4, 1) == E        # null y
    assert f(4, 4, A + 2, 4, B, 4, C, 4, 1) == gtg.GTG_ERR_MISALIGNED
    assert f(4, 4, A, 4, B, 4, A + 8, 4, 1) == gtg.GTG_ERR_ALIAS
    assert f(4, 4, A, 4, B, 4, B, 4, 1) == gtg.GTG_ERR_ALIAS
    assert f(0, 4, 0, 4, 0, 4, 0, 4, 1) == gtg.GTG_OK


def test_plan_validation_matches_the_call():
    with pytest.raises(gtg.GtgError) as e:
        gtg.plan_gemm("bf16", 4, 4, 8, A, 7, B, 4, C, 4)
    assert e.value.status == gtg.GTG_ERR_INVALID_VALUE
    assert gtg.plan_gemm("f32", 0, 4, 4, A, 4, B, 4, C, 4)["kernel"] == "none"


def test_epilogue_validation():
    E = gtg.GTG_ERR_INVALID_VALUE
    ep_bad_act = gtg.epilogue(0, 7)
    for fn in (gtg.gemm_f32_ex, gtg.gemm_tf32_ex, gtg.gemm_bf16_ex):
        assert fn(4, 4, 4, A, 4, B, 4, C, 4, ep_bad_act) == E
        # bias overlapping C, misaligned bias
        assert fn(4, 4, 4, A, 4, B, 4, C, 4, gtg.epilogue(C + 4, "relu")) == gtg.GTG_ERR_ALIAS
        assert fn(4, 4, 4, A, 4, B, 4, C, 4, gtg.epilogue(A + (1 << 20) + 2, "none")) == gtg.GTG_ERR_MISALIGNED
    assert gtg.gemv_f32_ex(4, 4, A, 4, B, 4, C, 4, 1, ep_bad_act) == E
    assert gtg.gemv_f32_ex(4, 4, A, 4, B, 4, C, 4, 1, gtg.epilogue(C + 8, "relu")) == gtg.GTG_ERR_ALIAS


def test_conv_validation():
    X, Wt, Y = A, B, C
    f = gtg.conv2d_nhwc
    E = gtg.GTG_ERR_INVALID_VALUE
    assert f("bf16", 1, 4, 4, 8, 8, 5, 5, 1, 1, 0, 0, 1, 1, X, Wt, Y) == E      # window larger than the image
    assert f("bf16", 1, 4, 4, 8, 8, 3, 3, 0, 1, 0, 0, 1, 1, X, Wt, Y) == E      # stride 0
    assert f("bf16", 1, 4, 4, 8, 8, 3, 3, 1, 1, -1, 0, 1, 1, X, Wt, Y) == E     # negative padding
    assert f("bf16", 1, 4, 4, 8, 8, 3, 3, 1, 1, 0, 0, 0, 1, X, Wt, Y) == E      # dilation 0
    assert f(9, 1, 4, 4, 8, 8, 3, 3, 1, 1, 0, 0, 1, 1, X, Wt, Y) == E
    assert f("bf16", 1, 4, 4, 8, 8, 3, 3, 1, 1, 0, 0, 1, 1, X + 1, Wt, Y) == gtg.GTG_ERR_MISALIGNED
    assert f("f32", 1, 4, 4, 8, 8, 3, 3, 1, 1, 0, 0, 1, 1, X, Wt, X + 64) == gtg.GTG_ERR_ALIAS
    assert f("bf16", 0, 4, 4, 8, 8, 3, 3, 1, 1, 0, 0, 1, 1, 0, 0, 0) == gtg.GTG_OK   # empty batch
