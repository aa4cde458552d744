"""The C-ABI library without a GPU: it builds, loads, exports every function
that include/ctc_packed.h declares, sizes workspaces, and rejects the
arguments the host can check before any CUDA call is made."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ctc_packed.h")


@pytest.fixture(scope="module")
def lib():
    from packed_sequence_ctc_gb300 import build as b

    path = b.build()
    import packed_sequence_ctc_gb300 as p

    return p.load_library(path)


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(ctc_packed_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["ctc_packed_workspace_size", "ctc_packed_forward", "ctc_packed_backward", "ctc_packed_read_status",
              "ctc_packed_status_string"]:
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", lib._name], capture_output=True, text=True, check=True).stdout
    exported = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared_functions():
        assert name in exported, f"{name} is declared but not exported"
        assert hasattr(lib, name)


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "t.c"
    src.write_text('#include "ctc_packed.h"\nint main(void) { return (int)sizeof(ctc_packed_status); }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-c", str(src), "-o", str(tmp_path / "t.o"),
                    "-I", os.path.join(ROOT, "include"), "-I", "/usr/local/cuda/include"], check=True)


def test_workspace_size(lib):
    f = lib.ctc_packed_workspace_size
    n = f(38400, 64, 200, 8193, 1)
    # two state-row buffers of T_total rows (12 offset ints + 404 state ints),
    # the emission matrix (T_total x 201 entries of 16 bytes) and the
    # backward's class sums (T_total x 201 entries of 8 bytes) dominate
    big = 2 * 38400 * (12 + 404) * 4 + 38400 * 201 * 16 + 38400 * 201 * 8
    assert big <= n < big + 4 * 2**20
    assert f(0, 0, 0, 1, 0) > 0
    assert f(-1, 1, 1, 4, 0) == 0
    assert f(10, 1, 1, 0, 0) == 0
    assert f(10, 1, 1, (1 << 20) + 1, 0) == 0  # unsupported D
    assert f(10, 1, 1, 32769, 0) > 0  # rows wider than any shared-memory tile are streamed in batches
    assert f(10, 1, 3840, 8, 0) == 0  # unsupported target bound
    assert f(10, 1, 1, 8, 7) == 0  # unknown dtype


def _fwd(lib, **kw):
    args = dict(lp=8, dtype=0, T=10, D=5, cu=16, ln=24, tg=32, tl=40, B=2, mtl=3, blank=0, zi=0, red=0, loss=48,
                ws=256, wsb=1 << 30, flags=0, stream=None)
    args.update(kw)
    return lib.ctc_packed_forward(args["lp"], args["dtype"], args["T"], args["D"], args["cu"], args["ln"], args["tg"],
                                  args["tl"], args["B"], args["mtl"], args["blank"], args["zi"], args["red"],
                                  args["loss"], args["ws"], args["wsb"], args["flags"], args["stream"])


def test_host_argument_checks_return_before_any_cuda_call(lib):
    INVALID, WORKSPACE, UNSUPPORTED = 1, 2, 4
    assert _fwd(lib, D=0) == INVALID
    assert _fwd(lib, blank=5) == INVALID
    assert _fwd(lib, blank=-1) == INVALID
    assert _fwd(lib, dtype=3) == INVALID
    assert _fwd(lib, red=5) == INVALID  # 0..4 are none, sum, mean, mean_batch, mean_volume
    assert _fwd(lib, B=-1) == INVALID
    assert _fwd(lib, cu=None) == INVALID
    assert _fwd(lib, loss=None) == INVALID
    assert _fwd(lib, lp=None) == INVALID
    assert _fwd(lib, lp=9) == INVALID  # misaligned float32 pointer
    assert _fwd(lib, flags=4) == INVALID
    assert _fwd(lib, ws=None) == WORKSPACE
    assert _fwd(lib, ws=128) == WORKSPACE  # not 256-byte aligned
    assert _fwd(lib, wsb=16) == WORKSPACE
    assert _fwd(lib, D=(1 << 20) + 1) == UNSUPPORTED
    assert _fwd(lib, mtl=3840) == UNSUPPORTED
    b = lib.ctc_packed_backward
    # grad overlapping log_probs
    assert b(4096, 0, 10, 5, 16, 24, 32, 40, 2, 3, 0, 0, 0, 48, 256, 1 << 30, 4096 + 20, None) == INVALID
    assert b(4096, 0, 10, 5, 16, 24, 32, 40, 2, 3, 0, 0, 0, None, 256, 1 << 30, 1 << 20, None) == INVALID
    assert lib.ctc_packed_read_status(None, None, None) == INVALID


def _fwd64(lib, **kw):
    args = dict(lp=8, T=10, D=5, cu=16, ln=24, tg=32, tl=40, B=2, mtl=3, blank=0, zi=0, red=0, loss=48,
                ws=256, wsb=1 << 30, flags=0, stream=None)
    args.update(kw)
    return lib.ctc_packed_forward_f64(args["lp"], args["T"], args["D"], args["cu"], args["ln"], args["tg"],
                                      args["tl"], args["B"], args["mtl"], args["blank"], args["zi"], args["red"],
                                      args["loss"], args["ws"], args["wsb"], args["flags"], args["stream"])


def test_float64_entry_points_check_before_any_cuda_call(lib):
    INVALID, WORKSPACE, UNSUPPORTED = 1, 2, 4
    F64 = 3
    n = lib.ctc_packed_workspace_size(1000, 4, 50, 30, F64)
    # alpha rows (12 bytes a state), emissions (16 bytes a label slot) and class sums (8 bytes) per frame
    assert n >= 1000 * 101 * 12 + 1000 * 51 * 16 + 1000 * 30 * 8
    assert 0 < lib.ctc_packed_workspace_size_loss_only(1000, 4, 50, 30, F64) < n
    assert lib.ctc_packed_workspace_size(1000, 4, 3840, 30, F64) == 0
    assert _fwd(lib, dtype=F64) == INVALID  # the generic entry points take no float64
    assert _fwd64(lib, lp=12) == INVALID  # misaligned float64 pointer
    assert _fwd64(lib, loss=None) == INVALID
    assert _fwd64(lib, red=5) == INVALID
    assert _fwd64(lib, blank=5) == INVALID
    assert _fwd64(lib, flags=4) == INVALID
    assert _fwd64(lib, D=(1 << 20) + 1) == UNSUPPORTED
    assert _fwd64(lib, mtl=3840) == UNSUPPORTED
    assert _fwd64(lib, ws=None) == WORKSPACE
    assert _fwd64(lib, wsb=16) == WORKSPACE
    b = lib.ctc_packed_backward_f64
    # grad overlapping log_probs; grad misaligned; no upstream gradient
    assert b(4096, 10, 5, 16, 24, 32, 40, 2, 3, 0, 0, 0, 48, 256, 1 << 30, 4096 + 40, None) == INVALID
    assert b(4096, 10, 5, 16, 24, 32, 40, 2, 3, 0, 0, 0, 48, 256, 1 << 30, (1 << 20) + 4, None) == INVALID
    assert b(4096, 10, 5, 16, 24, 32, 40, 2, 3, 0, 0, 0, None, 256, 1 << 30, 1 << 20, None) == INVALID


def test_status_strings(lib):
    for code in range(5):
        assert lib.ctc_packed_status_string(code)
    assert lib.ctc_packed_status_string(99) == b"unknown status"


def test_python_binding_fails_loudly_without_library(tmp_path):
    import packed_sequence_ctc_gb300 as p

    with pytest.raises(RuntimeError, match="no fallback"):
        p.load_library(str(tmp_path / "missing.so"))


def _fsa_fwd(lib, **kw):
    args = dict(lp=8, dtype=0, T=10, D=5, cu=16, ln=24, B=2, so=32, sw=40, fw=48, S=6, eo=56, ed=64, ew=72, E=4,
                ms=3, ml=2, zi=0, loss=80, ws=256, wsb=1 << 30, stream=None)
    args.update(kw)
    return lib.ctc_packed_fsa_forward(args["lp"], args["dtype"], args["T"], args["D"], args["cu"], args["ln"],
                                      args["B"], args["so"], args["sw"], args["fw"], args["S"], args["eo"],
                                      args["ed"], args["ew"], args["E"], args["ms"], args["ml"], args["zi"],
                                      args["loss"], args["ws"], args["wsb"], args["stream"])


def test_fsa_host_checks_return_before_any_cuda_call(lib):
    INVALID, WORKSPACE, UNSUPPORTED = 1, 2, 4
    assert _fsa_fwd(lib, D=0) == INVALID
    assert _fsa_fwd(lib, dtype=3) == INVALID
    assert _fsa_fwd(lib, B=-1) == INVALID
    assert _fsa_fwd(lib, ml=0) == INVALID  # max_labels below 1
    assert _fsa_fwd(lib, S=-1) == INVALID
    assert _fsa_fwd(lib, cu=None) == INVALID
    assert _fsa_fwd(lib, so=None) == INVALID
    assert _fsa_fwd(lib, ed=None) == INVALID  # edges announced but missing
    assert _fsa_fwd(lib, loss=None) == INVALID
    assert _fsa_fwd(lib, ms=0) == UNSUPPORTED
    assert _fsa_fwd(lib, ms=4097) == UNSUPPORTED  # more states than a shared-memory row holds
    assert _fsa_fwd(lib, D=16385) == UNSUPPORTED
    # states and labels whose per-frame shared-memory buffers exceed a CTA's
    assert _fsa_fwd(lib, ms=4096, ml=3700, D=16384) == UNSUPPORTED
    assert _fsa_fwd(lib, ms=2048, ml=5500, D=16384) == UNSUPPORTED
    assert _fsa_fwd(lib, ws=None) == WORKSPACE
    assert _fsa_fwd(lib, ws=128) == WORKSPACE  # not 256-byte aligned
    assert _fsa_fwd(lib, wsb=64) == WORKSPACE


def test_fsa_workspace_size():
    import packed_sequence_ctc_gb300 as pk
    from packed_sequence_ctc_gb300 import build as b

    lib = pk.load_library(b.build())
    f = lib.ctc_packed_fsa_workspace_size  # (T_total, B, num_states, num_edges, max_states, max_labels, D)
    assert f(100, 4, 20, 60, 0, 5, 10) == 0
    assert f(100, 4, 20, 60, 10, 0, 10) == 0
    assert f(100, 4, -1, 60, 10, 5, 10) == 0
    assert f(100, 4, 20, -1, 10, 5, 10) == 0
    assert f(100, 4, 20, 60, 10, 5, 16385) == 0
    n = f(1000, 4, 200, 600, 50, 20, 30)
    # alpha and beta rows (8 B x states each, extended range), label values and class sums (8 B x
    # min(labels, D) each) per frame, and per edge three 16-byte records and two positions at least
    assert n >= 1000 * 50 * 16 + 1000 * 20 * 16 + 1000 * 8 + 600 * (48 + 8)
    # a recursion's per-frame buffers (about 20 bytes a state and 36 a label up to 2048 states, 28
    # a label above) and the row kernel's two stages of a row (32 bytes a state, 28 a label) must
    # each fit a CTA's shared memory
    assert f(1000, 4, 200, 600, 2048, 5000, 16384) > 0
    assert f(1000, 4, 200, 600, 2048, 5500, 16384) == 0
    assert f(1000, 4, 200, 600, 4096, 3400, 16384) > 0
    assert f(1000, 4, 200, 600, 4096, 3600, 16384) == 0
    assert f(1000, 4, 200, 600, 50, 200, 30) < f(1000, 4, 200, 600, 50, 200, 300)  # class sums capped at D
    assert f(1000, 4, 200, 600, 50, 20, 30) < f(1000, 4, 200, 6000, 50, 20, 30)  # edge lists grow with edges
