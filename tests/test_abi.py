"""Host-side checks of the C ABI: the library builds, loads and exports every declared symbol;
argument errors are caught on the host before any CUDA call (runs without a GPU)."""
import ctypes

import pytest

import mixed_sliding_global_gb300 as g
from mixed_sliding_global_gb300 import binding

FAKE = 0x10000  # an aligned, never dereferenced stand-in for a device pointer


def lib():
    return g.library()


def test_library_exports_every_declared_symbol():
    lib()  # builds the library first when it is missing or older than its sources
    names = g.exported_symbols()
    assert {"gemma_kv_append", "gemma_attn_decode", "gemma_attn_prefill",
            "gemma_attn_workspace_size", "gemma_status_string", "gemma_abi_version"} <= set(names)
    raw = ctypes.CDLL(g.library_path())
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings_and_version():
    assert g.gemma_status_string(0) == "GEMMA_OK"
    assert g.gemma_status_string(-4) == "GEMMA_ERR_WORKSPACE"
    assert g.gemma_status_string(99) == "GEMMA_UNKNOWN_STATUS"
    assert g.gemma_abi_version() == 1


def _ptrs(*xs):
    return (ctypes.c_void_p * len(xs))(*xs)


def _i32(*xs):
    return (ctypes.c_int32 * len(xs))(*xs)


def decode(owner=(0,), layer=0, n_layers=None, max_seq_len=64, batch=1, kind=1, window=0, n_q=4,
           n_kv=1, d=64, k_eq_v=1, cap=64, scale=0.125, dtype=0, ws=None, ws_bytes=0,
           kc=(FAKE,), vc=(None,)):
    n_layers = len(owner) if n_layers is None else n_layers
    return lib().gemma_attn_decode(FAKE, FAKE, _ptrs(*kc), _ptrs(*vc), _i32(*owner), n_layers, layer,
                                   FAKE, max_seq_len, batch, kind, window, n_q, n_kv, d, k_eq_v,
                                   cap, scale, dtype, ws, ws_bytes, None, None)


INVALID, UNSUPPORTED, CAPACITY = -1, -2, -3


@pytest.mark.parametrize("kwargs,status", [
    (dict(owner=(1,)), INVALID),                         # owner after the layer
    (dict(owner=(0, 0), layer=2), INVALID),              # layer out of range
    (dict(owner=(0, 0, 1), layer=2, kc=(FAKE, None, None)), INVALID),  # owner that is shared
    (dict(n_q=6, n_kv=4), INVALID),                      # n_q not a multiple of n_kv
    (dict(n_q=64, n_kv=2), UNSUPPORTED),                 # group of 32
    (dict(d=96), UNSUPPORTED),
    (dict(kind=0, window=0), INVALID),                   # sliding without a window
    (dict(kind=2), INVALID),
    (dict(max_seq_len=65), CAPACITY),
    (dict(max_seq_len=0), INVALID),
    (dict(k_eq_v=0), INVALID),                           # V cache missing
    (dict(kc=(None,)), INVALID),
    (dict(kc=(FAKE + 8,)), INVALID),                     # misaligned cache
    (dict(dtype=5), INVALID),
    (dict(scale=float("nan")), INVALID),
    (dict(scale=0.0), INVALID),
    (dict(scale=-0.5), INVALID),
    (dict(batch=-1), INVALID),
])
def test_decode_argument_errors(kwargs, status):
    assert decode(**kwargs) == status


@pytest.mark.parametrize("softcap,status", [(float("nan"), INVALID), (float("inf"), INVALID),
                                            (-1.0, INVALID)])
def test_softcap_argument_errors(softcap, status):
    """The soft-cap entry point rejects a negative or non-finite cap on the host."""
    st = lib().gemma_attn_softcap(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, 64, 1,
                                  1, 1, 0, 4, 1, 64, 1, 64, 0.125, softcap, 0, None, 0, None, None)
    assert st == status


def test_softcap_empty_batch_is_ok():
    assert lib().gemma_attn_softcap(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, 64,
                                    1, 0, 1, 0, 4, 1, 64, 1, 64, 0.125, 30.0, 0, None, 0, None,
                                    None) == 0


def test_bucket_entry_points_need_n_real():
    """The padded-bucket entry points reject a missing n_real array on the host."""
    assert lib().gemma_kv_append_bucket(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE,
                                        None, 1, 4, 1, 64, 64, 1, 0, None, None) == INVALID
    assert lib().gemma_attn_prefill_bucket(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0,
                                           FAKE, None, 64, 4, 1, 1, 0, 4, 1, 64, 1, 64, 0.125, 0,
                                           None, 0, None, None) == INVALID
    assert lib().gemma_attn_prefill_bucket(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0,
                                           FAKE, FAKE, 64, 4, 0, 1, 0, 4, 1, 64, 1, 64, 0.125, 0,
                                           None, 0, None, None) == 0   # empty batch


@pytest.mark.parametrize("cap,window,status", [(1000, 512, UNSUPPORTED),   # not a multiple of 128
                                                (512, 640, CAPACITY)])        # smaller than the window
def test_ring_capacity_checks(cap, window, status):
    """A ring cache (kind 2) needs a capacity that is a multiple of 128 and holds the window."""
    assert decode(kind=2, window=window, cap=cap, max_seq_len=4096, k_eq_v=0,
                  vc=(FAKE,)) == status


def test_ring_prefill_needs_window_plus_new_tokens():
    st = lib().gemma_attn_prefill(FAKE, FAKE, _ptrs(FAKE), _ptrs(FAKE), _i32(0), 1, 0, FAKE, 4096,
                                  130, 1, 2, 1024, 4, 1, 64, 0, 1152, 0.125, 0, None, 0, None,
                                  None)
    assert st == CAPACITY   # 1152 < 1024 + 130 - 1


def test_empty_batch_is_ok_without_touching_the_device():
    assert decode(batch=0) == 0
    assert lib().gemma_attn_prefill(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, 64,
                                    0, 1, 1, 0, 4, 1, 64, 1, 64, 0.1, 0, None, 0, None, None) == 0


def test_append_argument_errors_and_shared_no_op():
    f = lib().gemma_kv_append
    # shared layer: OK, nothing to do
    assert f(_ptrs(FAKE, None), _ptrs(None, None), _i32(0, 0), 2, 1, FAKE, None, FAKE, 1, 1, 1, 64,
             64, 1, 0, None, None) == 0
    # n_new beyond capacity
    assert f(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE, 1, 65, 1, 64, 64, 1, 0,
             None, None) == CAPACITY
    # V cache missing without k_eq_v
    assert f(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, FAKE, FAKE, 1, 1, 1, 64, 64, 0, 0,
             None, None) == INVALID
    assert f(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE, 1, 1, 1, 80, 64, 1, 0,
             None, None) == UNSUPPORTED
    # empty
    assert f(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE, 0, 1, 1, 64, 64, 1, 0,
             None, None) == 0


def test_workspace_size_rejects_bad_arguments():
    assert lib().gemma_attn_workspace_size(1, 1, 0, 6, 4, 64, 64, 1) == ctypes.c_size_t(-1).value
    assert lib().gemma_attn_workspace_size(0, 1, 0, 4, 1, 64, 64, 1) == 0
    with pytest.raises(ValueError):
        g.gemma_attn_workspace_size(1, 1, 0, 4, 1, 96, 64, 1)


def test_binding_has_no_fallback():
    # every computing entry point of the binding goes through the shared library
    src = open(binding.__file__).read()
    assert "oracle" not in src and "torch.nn.functional" not in src


@pytest.mark.parametrize("args,status", [
    ((FAKE, 1, 4, 0, float("nan")), INVALID), ((FAKE, 1, 4, 0, -1.0), INVALID),
    ((FAKE, 1, 0, 0, 30.0), INVALID), ((FAKE, -1, 4, 0, 30.0), INVALID),
    ((FAKE, 1, 4, 7, 30.0), INVALID), ((None, 1, 4, 0, 30.0), INVALID),
    ((FAKE + 8, 1, 4, 0, 30.0), INVALID), ((FAKE, 0, 4, 0, 30.0), 0),
])
def test_logit_argument_errors(args, status):
    """The logit soft-cap / argmax entry point rejects bad arguments on the host."""
    logits, batch, vocab, dtype, cap = args
    assert lib().gemma_logit_softcap_argmax(logits, batch, vocab, dtype, cap, None, FAKE, None, 0,
                                            None) == status
    assert lib().gemma_logit_softcap_argmax(FAKE, 1, 4, 0, 30.0, FAKE + 4, FAKE, None, 0,
                                            None) == INVALID   # misaligned capped output
    assert lib().gemma_logit_workspace_size(-1, 4) == ctypes.c_size_t(-1).value
    assert lib().gemma_logit_workspace_size(1, 0) == ctypes.c_size_t(-1).value
    assert lib().gemma_logit_workspace_size(0, 4) == 0


def test_paged_argument_checks():
    """The paged entry points reject a page size that is not a multiple of 128, empty pools and
    ring kinds on the host."""
    f = lib().gemma_attn_paged
    base = dict(max_pages=4, page_size=128, n_pages=8, kind=1, msl=64)

    def call(**kw):
        a = {**base, **kw}
        return f(FAKE, FAKE, _ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, FAKE, a["max_pages"],
                 a["page_size"], a["n_pages"], a["msl"], 1, 1, a["kind"], 0, 4, 1, 64, 1, 0.125,
                 0, None, None, None, None, 0, None, None)
    assert call(page_size=100) == UNSUPPORTED
    assert call(page_size=64) == UNSUPPORTED
    assert call(n_pages=0) == INVALID
    assert call(max_pages=0) == INVALID
    assert call(kind=2) == INVALID
    assert call(msl=513) == CAPACITY   # beyond max_pages * page_size
    a = lib().gemma_kv_append_paged
    assert a(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE, None, 4, 128, 8, 1, 1,
             1, 64, 1, 0, None, None) == INVALID   # block table missing
    assert a(_ptrs(FAKE), _ptrs(None), _i32(0), 1, 0, FAKE, None, FAKE, FAKE, 4, 130, 8, 1, 1,
             1, 64, 1, 0, None, None) == UNSUPPORTED
    assert lib().gemma_attn_workspace_size_paged(1, 2, 512, 4, 1, 64, 64, 1) == \
        ctypes.c_size_t(-1).value


def test_binding_signatures_match_the_header():
    """Every prototype in include/gemma_attn.h has as many parameters as the binding's ctypes
    signature of the same name (an ABI change cannot silently misalign the marshalling)."""
    import re
    with open(binding._build.HEADER) as f:
        text = f.read()
    protos = re.findall(r"^\s*(?:int|size_t|const char\*)\s+(gemma_\w+)\s*\(([^)]*)\)\s*;",
                        text, re.M | re.S)
    assert len(protos) == len(g.exported_symbols())
    for name, params in protos:
        params = params.strip()
        n = 0 if params in ("", "void") else params.count(",") + 1
        assert name in binding._SIGNATURES, name
        assert len(binding._SIGNATURES[name][1]) == n, (name, n, len(binding._SIGNATURES[name][1]))


def decode_static(owner=(0,), layer=0, max_seq_len=64, batch=1, kind=1, window=0, n_q=4, n_kv=1,
                  d=64, k_eq_v=1, cap=64, scale=0.125, dtype=0, kc=(FAKE,), vc=(None,)):
    return lib().gemma_attn_decode_static(FAKE, FAKE, _ptrs(*kc), _ptrs(*vc), _i32(*owner),
                                          len(owner), layer, FAKE, max_seq_len, batch, kind,
                                          window, n_q, n_kv, d, k_eq_v, cap, scale, dtype, None,
                                          None)


@pytest.mark.parametrize("kwargs,status", [
    (dict(d=96), UNSUPPORTED),
    (dict(n_q=64, n_kv=2), UNSUPPORTED),                 # group of 32
    (dict(owner=(1,)), INVALID),
    (dict(max_seq_len=65), CAPACITY),
    (dict(k_eq_v=0), INVALID),                           # V cache missing
    (dict(scale=0.0), INVALID),
    (dict(batch=-1), INVALID),
])
def test_static_decode_reports_the_statuses_of_the_workspace_decode(kwargs, status):
    """The allocation-free decode returns what gemma_attn_decode returns for the same bad
    arguments (no GPU is touched: every check fails on the host first)."""
    assert decode_static(**kwargs) == status
    assert decode(**kwargs) == status


def test_static_decode_empty_batch_is_ok():
    assert decode_static(batch=0) == 0
