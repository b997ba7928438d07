"""Host-side checks of the C ABI, runnable without a GPU: the library loads,
exports every entry point declared in include/*.h, its parameter block has
the declared layout, argument errors are reported before any CUDA call, and
the workspace stays O(rows) (the pages' one-logits-tensor memory rule)."""
import ctypes
import glob
import json
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared_functions():
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        for m in re.finditer(r"\b([a-z_][a-z0-9_]*)\s*\(", text):
            name = m.group(1)
            # declarations only: return type precedes the name on the same statement
            before = text[:m.start()].rstrip()
            if before.endswith(("*", "ce_status", "void", "char", "int", "size_t")) or re.search(
                    r"(ce_status|const char \*|void|int32_t|size_t)\s*\**\s*$", before):
                names.add(name)
    return sorted(n for n in names if n not in {"sizeof"})


@pytest.fixture(scope="module")
def lib():
    import softmax_cross_entropy_pass_gb300 as ce
    return ce


def test_header_declares_entry_points():
    names = _declared_functions()
    for n in ("ce_forward", "ce_backward", "ce_fwd_bwd", "ce_scale_grad", "ce_workspace_size",
              "ce_get_status", "ce_fused_plan", "ce_version", "ce_status_string"):
        assert n in names, n


def test_library_exports_every_declared_symbol(lib):
    so = ctypes.CDLL(lib.LIB_PATH)
    missing = [n for n in _declared_functions() if not hasattr(so, n)]
    assert not missing, missing


def test_version_and_status_strings(lib):
    assert "sm_103a" in lib.version()
    assert lib._lib.ce_status_string(1) == b"CE_ERR_INVALID_ARG"


def test_params_layout(lib):
    P = lib.ce_params
    assert ctypes.sizeof(P) == 80
    assert P.class_weight.offset == 32 and P.label_smoothing.offset == 40 and P.reserved.offset == 60
    assert P.softcap.offset == 64 and P.z_loss.offset == 68 and P.accuracy.offset == 72


def _params(lib, **kw):
    p = lib.ce_params()
    p.n_rows, p.vocab, p.ld = kw.get("n_rows", 4), kw.get("vocab", 10), kw.get("ld", 10)
    p.label_smoothing = kw.get("eps", 0.0)
    p.dtype, p.reduction = kw.get("dtype", 1), kw.get("reduction", 1)
    p.variant, p.reserved = kw.get("variant", 0), kw.get("reserved", 0)
    p.softcap, p.z_loss = kw.get("softcap", 0.0), kw.get("z_loss", 0.0)
    return p


@pytest.mark.parametrize("bad", [dict(vocab=0), dict(ld=5), dict(n_rows=-1), dict(eps=1.5),
                                 dict(eps=float("nan")), dict(dtype=7), dict(reduction=9),
                                 dict(reserved=1), dict(softcap=-1.0), dict(z_loss=float("inf"))])
def test_invalid_params_rejected_on_host(lib, bad):
    p = _params(lib, **bad)
    fake = ctypes.c_void_p(0x1000)
    st = lib._lib.ce_fwd_bwd(ctypes.byref(p), fake, fake, fake, None, ctypes.c_void_p(0x100000), 1 << 20, None)
    assert st == lib.CE_ERR_INVALID_ARG


def test_workspace_errors_rejected_on_host(lib):
    p = _params(lib)
    fake = ctypes.c_void_p(0x1000)
    # NULL, misaligned and too small workspaces
    for ws, nb in ((None, 1 << 20), (ctypes.c_void_p(0x100010), 1 << 20), (ctypes.c_void_p(0x100000), 16)):
        st = lib._lib.ce_fwd_bwd(ctypes.byref(p), fake, fake, fake, None, ws, nb, None)
        assert st == lib.CE_ERR_WORKSPACE


def test_workspace_is_o_rows_and_far_below_one_logits_tensor(lib):
    """The pages' peak memory for BT=8192, V=128256 bf16 is the logits tensor
    alone (2004 MB); the library's scratch must be a rounding error on it."""
    gold = json.load(open(os.path.join(ROOT, "tests", "golden", "peak_memory_mb.json")))
    mb = gold["bf16_vocab_sweep_bt8192"]["128256"]
    ws = lib.ce_workspace_size(8192)
    assert ws <= 20 * 8192 + 512
    assert ws / 2 ** 20 < 0.001 * mb
    assert lib.ce_workspace_size(16384) - lib.ce_workspace_size(8192) == 20 * 8192


def test_automatic_path_choice_is_host_logic(lib):
    """ce_select_variant (no GPU work): every row layout and every option set
    takes the stream kernel; explicit variants are returned as asked."""
    out = ctypes.c_int32()
    p = _params(lib, n_rows=4, vocab=128256, ld=128256)
    assert lib._lib.ce_select_variant(ctypes.byref(p), ctypes.c_void_p(0x10000), ctypes.byref(out)) == 0
    assert out.value == lib.VARIANTS["stream"]
    p = _params(lib, n_rows=4, vocab=1001, ld=1001)   # 2002-byte rows: not 16-byte aligned
    assert lib._lib.ce_select_variant(ctypes.byref(p), ctypes.c_void_p(0x10000), ctypes.byref(out)) == 0
    assert out.value == lib.VARIANTS["stream"]
    p = _params(lib, n_rows=4, vocab=128256, ld=128256)
    assert lib._lib.ce_select_variant(ctypes.byref(p), ctypes.c_void_p(0x10008), ctypes.byref(out)) == 0
    assert out.value == lib.VARIANTS["stream"]
    p = _params(lib, n_rows=4, vocab=128256, ld=128256)
    p.softcap = 30.0
    assert lib._lib.ce_select_variant(ctypes.byref(p), ctypes.c_void_p(0x10000), ctypes.byref(out)) == 0
    assert out.value == lib.VARIANTS["stream"]
    p = _params(lib, variant=lib.VARIANTS["split"])
    assert lib._lib.ce_select_variant(ctypes.byref(p), ctypes.c_void_p(0x10000), ctypes.byref(out)) == 0
    assert out.value == lib.VARIANTS["split"]


def test_gemm_and_flce_argument_errors_on_host(lib):
    """Misaligned bias pointers and unknown fused-linear variant bits are
    refused before any CUDA call."""
    L = lib._lib
    fake = ctypes.c_void_p(0x100000)
    st = L.ce_gemm_bf16(128, 256, 64, fake, 64, 0, fake, 64, 0, 0, fake, 256, ctypes.c_void_p(0x100004), None)
    assert st == 1
    p = lib.ce_params()
    p.n_rows, p.vocab, p.ld, p.dtype, p.reduction, p.ignore_index = 64, 1024, 1024, 1, 1, -100
    for variant, bias in ((4, None), (0, ctypes.c_void_p(0x100008))):
        p.variant = variant
        st = L.flce_fwd_bwd(ctypes.byref(p), 64, fake, fake, bias, fake, fake, None, fake, fake, fake, 64,
                            ctypes.c_void_p(0x200000), 1 << 40, None)
        assert st == 1, (variant, bias)


def test_flce_workspace_by_variant(lib):
    """The compacted path adds a copy of hidden (BT x H bf16) and a few bytes
    per row; the statistics path adds 16 bytes (row state) and 8 bytes
    (argmax for the token accuracy) per row and 256-column tile of a chunk,
    plus 32 bytes per chunk row; all stay far below the logits."""
    BT, H, V, C = 8192, 4096, 128256, 4096
    base = lib.flce_workspace_size(BT, H, V, C, dense=True, ce_cluster=True)
    compact = lib.flce_workspace_size(BT, H, V, C, dense=False, ce_cluster=True)
    stats = lib.flce_workspace_size(BT, H, V, C, dense=True, ce_cluster=False)
    both = lib.flce_workspace_size(BT, H, V, C)
    assert compact - base >= BT * H * 2 and compact - base <= BT * H * 2 + BT * 32 + 8192
    tiles = (V + 255) // 256
    assert stats - base >= C * tiles * 24 + C * 32 and stats - base <= C * tiles * 24 + C * 32 + 4096
    assert both == base + (compact - base) + (stats - base)
    assert base >= C * V * 6                       # fp32 logits chunk + bf16 dZ chunk


def test_logits_not_element_aligned_rejected_on_host(lib):
    """A bf16 logits pointer at an odd address is refused by every entry point."""
    L = lib._lib
    p = _params(lib, n_rows=4, vocab=1000, ld=1000)
    fake, odd = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x100001)
    ws, nb = ctypes.c_void_p(0x200000), 1 << 20
    assert L.ce_fwd_bwd(ctypes.byref(p), odd, fake, fake, None, ws, nb, None) == 1
    assert L.ce_forward(ctypes.byref(p), odd, fake, fake, fake, ws, nb, None) == 1
    assert L.ce_backward(ctypes.byref(p), odd, fake, fake, None, ws, nb, None) == 1


def test_from_host_argument_errors_on_host(lib):
    """ce_fwd_bwd_from_host refuses n_parts < 1, the same stream for copies and
    kernels, a variant, and the options, before any CUDA call."""
    L = lib._lib
    fake, ws = ctypes.c_void_p(0x100000), ctypes.c_void_p(0x200000)
    p = _params(lib, n_rows=4, vocab=1000, ld=1000)
    s1, s2 = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    assert L.ce_fwd_bwd_from_host(ctypes.byref(p), fake, fake, fake, fake, None, ws, 1 << 20, s1, s2, 0) == 1
    assert L.ce_fwd_bwd_from_host(ctypes.byref(p), fake, fake, fake, fake, None, ws, 1 << 20, s1, s1, 4) == 1
    p.variant = 4
    assert L.ce_fwd_bwd_from_host(ctypes.byref(p), fake, fake, fake, fake, None, ws, 1 << 20, s1, s2, 4) == 1
    p = _params(lib, n_rows=4, vocab=1000, ld=1000, softcap=10.0)
    assert L.ce_fwd_bwd_from_host(ctypes.byref(p), fake, fake, fake, fake, None, ws, 1 << 20, s1, s2, 4) == 2
