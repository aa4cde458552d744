"""Host-side behaviour of the Python binding that needs no GPU: argument
checks of the autograd wrapper before any launch, the status-bit messages,
and that the library's entry points are bound with the arity the header
declares (a call with a wrong argument count would fail in ctypes)."""

import re
import os

import pytest
import torch

import packed_sequence_ctc_gb300 as pk

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_wrapper_rejects_bad_arguments_before_any_launch():
    lp = torch.zeros(10, 5)
    cu = torch.tensor([0, 6, 10])
    ln = torch.tensor([6, 4])
    tg = torch.tensor([1, 2, 3])
    tl = torch.tensor([2, 1])
    with pytest.raises(ValueError, match="unexpected reduction"):
        pk.packed_ctc_loss(lp, cu, ln, tg, tl, blank=0, reduction="average")
    with pytest.raises(ValueError, match="blank"):
        pk.packed_ctc_loss(lp, cu, ln, tg, tl, blank=5, max_target_len=2)
    with pytest.raises(TypeError, match="float64"):
        pk.packed_ctc_loss(lp.to(torch.int32), cu, ln, tg, tl, blank=0, max_target_len=2)  # no integer path
    with pytest.raises(ValueError, match="CUDA"):
        pk.packed_ctc_loss(lp, cu, ln, tg, tl, blank=0, max_target_len=2)  # a CPU tensor: no CPU path


def test_reduction_and_flag_codes_match_the_header():
    text = open(os.path.join(ROOT, "include", "ctc_packed.h")).read()
    enum = dict((name.lower(), int(v)) for name, v in re.findall(r"CTC_PACKED_(NONE|SUM|MEAN|MEAN_BATCH|MEAN_VOLUME)"
                                                                  r"\s*=\s*(\d+)", text))
    assert enum == pk.REDUCTION_CODES
    assert int(re.search(r"#define CTC_PACKED_FLAG_LOSS_ONLY (0x\w+)u", text).group(1), 16) == pk.FLAG_LOSS_ONLY
    assert int(re.search(r"#define CTC_PACKED_FLAG_LOGITS (0x\w+)u", text).group(1), 16) == pk.FLAG_LOGITS
    bits = {int(v, 16) for v in re.findall(r"#define CTC_PACKED_DEV_\w+ (0x\w+)u", text)}
    assert bits == set(pk.DEVICE_STATUS_BITS)


def test_entry_points_are_bound_with_the_declared_arity():
    from packed_sequence_ctc_gb300 import build as b

    lib = pk.load_library(b.build())
    text = open(os.path.join(ROOT, "include", "ctc_packed.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    for name, params in re.findall(r"\b(ctc_packed_\w+)\s*\(([^;{]*?)\)\s*;", text, flags=re.S):
        n = 0 if params.strip() in ("", "void") else params.count(",") + 1
        fn = getattr(lib, name)
        assert fn.argtypes is not None and len(fn.argtypes) == n, name


def test_fsa_wrappers_check_their_tensors_before_any_call():
    import workloads

    lp = torch.zeros(8, 4)
    cu = torch.tensor([0, 8], dtype=torch.int32)
    ln = torch.tensor([8], dtype=torch.int32)
    fsa = workloads.pack_fsas([workloads.random_fsa(3, 6, 4, seed=0)])
    ws = torch.empty(1 << 20, dtype=torch.uint8)
    loss = torch.empty(1)
    pk.ctc_packed_fsa_forward  # bound
    bad_edges = (fsa[0], fsa[1], fsa[2], fsa[3], fsa[4].long(), fsa[5])
    with pytest.raises(TypeError, match="edges"):
        pk.ctc_packed_fsa_forward(lp, cu, ln, bad_edges, 3, 4, False, loss, ws)
    flat = (fsa[0], fsa[1], fsa[2], fsa[3], fsa[4].reshape(-1), fsa[5])
    with pytest.raises(ValueError, match="shape"):
        pk.ctc_packed_fsa_forward(lp, cu, ln, flat, 3, 4, False, loss, ws)
    short = (fsa[0], fsa[1], fsa[2], fsa[3], fsa[4], fsa[5][:-1])
    with pytest.raises(ValueError, match="edge_weight"):
        pk.ctc_packed_fsa_forward(lp, cu, ln, short, 3, 4, False, loss, ws)
    with pytest.raises(TypeError, match="cu_seqlens"):
        pk.ctc_packed_fsa_forward(lp, cu.long(), ln, fsa, 3, 4, False, loss, ws)


def test_noalloc_wrapper_checks_its_tensors_before_any_launch():
    lp = torch.zeros(10, 5)
    cu = torch.tensor([0, 6, 10], dtype=torch.int32)
    ln = torch.tensor([6, 4], dtype=torch.int32)
    tg = torch.tensor([1, 2, 3], dtype=torch.int32)
    tl = torch.tensor([2, 1], dtype=torch.int32)
    loss = torch.zeros(2)
    with pytest.raises(TypeError, match="log_probs"):
        pk.ctc_packed_forward_noalloc(lp.double(), cu, ln, tg, tl, 0, False, "none", loss, 2)
    with pytest.raises(TypeError, match="log_probs"):
        pk.ctc_packed_forward_noalloc(lp.t(), cu, ln, tg, tl, 0, False, "none", loss, 2)  # not contiguous
    with pytest.raises(TypeError, match="cu_seqlens"):
        pk.ctc_packed_forward_noalloc(lp, cu.long(), ln, tg, tl, 0, False, "none", loss, 2)
    with pytest.raises(TypeError, match="targets"):
        pk.ctc_packed_forward_noalloc(lp, cu, ln, tg[::2], tl, 0, False, "none", loss, 2)
    with pytest.raises(TypeError, match="loss"):
        pk.ctc_packed_forward_noalloc(lp, cu, ln, tg, tl, 0, False, "none", loss.double(), 2)
