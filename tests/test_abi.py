"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/flce.h declares, sizes its workspace independently of
N beyond one chunk, and rejects bad arguments with status codes before any
device work."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    import __graft_entry__
    __graft_entry__.build()
    from linear_cross_entropy_02_gb300 import _lib
    return _lib.lib()


def _declared():
    with open(os.path.join(ROOT, "include", "flce.h")) as f:
        src = f.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(flce_[a-z_]+)\s*\(", src)))


def test_exports_every_declared_symbol(L):
    names = _declared()
    assert "flce_forward_backward" in names and "flce_ce_only" in names and "flce_forward" in names
    for n in names:
        assert hasattr(L, n), n
    from linear_cross_entropy_02_gb300 import _lib
    assert sorted(_lib.EXPORTED) == names


def test_header_constants_match_binding():
    from linear_cross_entropy_02_gb300 import _lib
    with open(os.path.join(ROOT, "include", "flce.h")) as f:
        src = f.read()
    for name, val in re.findall(r"#define (FLCE_[A-Z0-9_]+) (\d+)", src):
        assert getattr(_lib, name) == int(val), name


def _params(L, N=4096, H=512, V=4096, **kw):
    from linear_cross_entropy_02_gb300._lib import FlceParams
    p = FlceParams()
    L.flce_default_params(ctypes.byref(p))
    p.n_rows, p.hidden, p.vocab = N, H, V
    for k, v in kw.items():
        setattr(p, k, v)
    return p


def test_default_params(L):
    p = _params(L)
    assert p.out_mult == 1.0 and p.softcap == 0.0 and p.ignore_index == -100
    assert p.grad_scale == 1.0 and p.reduction == 0 and p.chunk_rows == 0


def test_workspace_independent_of_n_beyond_a_chunk(L):
    sizes = []
    for N in (8192, 16384, 32768, 65536):
        p = _params(L, N=N, H=7168, V=129280, chunk_rows=8192)
        sizes.append(L.flce_workspace_size(ctypes.byref(p), 2, 1, 1))
    assert len(set(sizes)) == 1 and sizes[0] > 0
    # transient is O(C V): far below a [N, V] fp32 logits tensor at N = 32768
    assert sizes[0] < 32768 * 129280 * 4
    # CE-only keeps no logits at all: only per-tile statistics
    p = _params(L, N=131072, H=4096, V=151936)
    ce = L.flce_workspace_size(ctypes.byref(p), 0, 0, 0)
    assert 0 < ce < 100e6
    # the backward GEMMs read W, dz and h in place (MN-major tiles): no transposed
    # copies, so a frozen W costs no less than a trained one and the K-major
    # cross-check (explicit transposes) costs more
    p = _params(L, N=32768, H=7168, V=129280)
    both = L.flce_workspace_size(ctypes.byref(p), 2, 1, 1)
    assert L.flce_workspace_size(ctypes.byref(p), 2, 1, 0) == both
    pk = _params(L, N=32768, H=7168, V=129280, flags=4)
    assert L.flce_workspace_size(ctypes.byref(pk), 2, 1, 1) > both + 129280 * 7168 * 2
    # cross-entropy on materialised logits keeps only per-tile statistics
    pc = _params(L, N=131072, H=0, V=151936)
    assert 0 < L.flce_workspace_size(ctypes.byref(pc), 3, 0, 0) < 100e6


def test_default_chunk_fills_the_gemm_waves(L):
    """chunk_rows = 0 on the stored-logits backward: 8192 rows unless another
    multiple of 256 up to 10240 fills the GEMMs' waves better. On the frozen
    131072 x 4096 x 151936 head with grad_h only that is 9728 rows: 38 units of
    256 rows x 16 column tiles = 608 tiles, exactly 4 waves on 152 SMs. The
    DSV3, Llama and Muse heads keep 8192, and so do the recompute backward and
    an explicit chunk size."""
    def ws(N, H, V, gw, chunk=0, flags=0):
        p = _params(L, N=N, H=H, V=V, chunk_rows=chunk, flags=flags)
        return L.flce_workspace_size(ctypes.byref(p), 2, 1, int(gw))
    assert ws(131072, 4096, 151936, False) == ws(131072, 4096, 151936, False, 9728)
    assert ws(131072, 4096, 151936, False) > ws(131072, 4096, 151936, False, 8192)
    for N, H, V in ((32768, 7168, 129280), (8192, 4096, 128256), (8192, 6656, 202048)):
        assert ws(N, H, V, True) == ws(N, H, V, True, 8192), (N, H, V)
    assert ws(131072, 4096, 151936, False, flags=8) == ws(131072, 4096, 151936, False, 8192, flags=8)

    def rows(N, H, V, gw, mode=2, chunk=0, flags=0):
        p = _params(L, N=N, H=H, V=V, chunk_rows=chunk, flags=flags)
        return L.flce_chunk_rows(ctypes.byref(p), mode, 1, int(gw))
    assert rows(131072, 4096, 151936, False) == 9728
    assert rows(32768, 7168, 129280, True) == 8192
    assert rows(131072, 4096, 151936, False, mode=0) == 8192           # CE-only
    assert rows(131072, 4096, 151936, False, flags=8) == 8192          # recompute backward
    assert rows(300, 64, 100, True) == 384 and rows(300, 64, 100, True, chunk=200) == 256
    assert rows(300, 64, 100, True, chunk=100000) == 384                # at most N rounded up
    assert rows(300, 12, 100, True) == 0                                # H % 8 != 0


@pytest.mark.parametrize("field,value", [("hidden", 0), ("vocab", 0), ("n_rows", -1), ("softcap", -1.0),
                                         ("reduction", 7), ("chunk_rows", -5), ("ld_h", 100)])
def test_workspace_size_rejects_bad_params(L, field, value):
    p = _params(L, **{field: value})
    assert L.flce_workspace_size(ctypes.byref(p), 2, 1, 1) == 0


def test_host_errors_before_any_device_work(L):
    from linear_cross_entropy_02_gb300 import _lib as B
    fake = ctypes.c_void_p(1 << 20)          # never dereferenced: every call below fails on the host
    p = _params(L)
    # too-small workspace
    rc = L.flce_forward_backward(ctypes.byref(p), fake, fake, fake, fake, None, None, fake, fake, fake, 256, None)
    assert rc == B.FLCE_ERR_WORKSPACE
    # null loss
    rc = L.flce_ce_only(ctypes.byref(p), fake, fake, fake, None, None, fake, 1 << 40, None)
    assert rc == B.FLCE_ERR_ARG
    # misaligned h
    rc = L.flce_ce_only(ctypes.byref(p), ctypes.c_void_p((1 << 20) + 2), fake, fake, fake, None, fake, 1 << 40,
                        None)
    assert rc == B.FLCE_ERR_ALIGN
    # H not a multiple of 8
    p2 = _params(L, H=100)
    rc = L.flce_ce_only(ctypes.byref(p2), fake, fake, fake, fake, None, fake, 1 << 40, None)
    assert rc == B.FLCE_ERR_ALIGN
    # negative softcap
    p3 = _params(L, softcap=-2.0)
    rc = L.flce_forward(ctypes.byref(p3), fake, fake, fake, fake, None, None, None, fake, 1 << 40, None)
    assert rc == B.FLCE_ERR_ARG
    # null params
    assert L.flce_ce_only(None, fake, fake, fake, fake, None, fake, 1 << 40, None) == B.FLCE_ERR_ARG


def test_status_strings(L):
    for code in (0, 1, 2, 3, 4, 5, 16, 32, 48, 64, 999):
        s = L.flce_status_string(code)
        assert isinstance(s, bytes) and len(s) > 0
    assert L.flce_status_string(32) == b"bounded device wait timed out"
    assert b"non-finite" in L.flce_status_string(64)


def test_kernel_names(L):
    from linear_cross_entropy_02_gb300 import _lib as B
    names = [L.flce_kernel_name(i).decode() for i in range(B.FLCE_NUM_KERNELS)]
    assert names[1] == "fwd_gemm_stats" and names[4] == "grad_h_gemm" and names[5] == "grad_W_gemm"
    assert names[14:] == ["scale_gradient", "vp_merge", "split_tf32"]
    assert len(set(names)) == len(names) and "unknown" not in names
    assert L.flce_kernel_name(B.FLCE_NUM_KERNELS) == b"unknown"
    assert L.flce_kernel_name(99) == b"unknown"


def test_host_buffer_entries_host_errors(L):
    """The host-buffer entry points reject bad arguments before touching the
    device or the host buffers (the pointers below are never dereferenced)."""
    from linear_cross_entropy_02_gb300 import _lib as B
    fake = ctypes.c_void_p(1 << 20)
    p = _params(L)
    need = L.flce_workspace_size(ctypes.byref(p), B.FLCE_MODE_FORWARD_BACKWARD_HOST, 1, 1)
    base = L.flce_workspace_size(ctypes.byref(p), B.FLCE_MODE_FORWARD_BACKWARD, 1, 1)
    # two chunks of h (bf16) and the labels on top of the device-input workspace
    assert need >= base + 2 * 4096 * 512 * 2 + 4096 * 8
    assert L.flce_workspace_size(ctypes.byref(p), B.FLCE_MODE_CE_ONLY_HOST, 0, 0) > \
        L.flce_workspace_size(ctypes.byref(p), B.FLCE_MODE_CE_ONLY, 0, 0)
    assert L.flce_workspace_size(ctypes.byref(p), 6, 0, 0) == 0             # unknown mode
    rc = L.flce_forward_backward_from_host(ctypes.byref(p), fake, fake, fake, fake, None, None, fake, fake, fake,
                                           need - 256, None, None)
    assert rc == B.FLCE_ERR_WORKSPACE
    rc = L.flce_forward_backward_from_host(ctypes.byref(p), fake, fake, fake, None, None, None, fake, fake, fake,
                                           need, None, None)
    assert rc == B.FLCE_ERR_ARG                                                  # no loss output
    ps = _params(L, flags=B.FLCE_FLAG_SIMT_GEMM)
    rc = L.flce_forward_backward_from_host(ctypes.byref(ps), fake, fake, fake, fake, None, None, fake, fake, fake,
                                           1 << 40, None, None)
    assert rc == B.FLCE_ERR_UNSUPPORTED
    pf = _params(L, dtype=B.FLCE_DTYPE_F32, flags=B.FLCE_FLAG_SIMT_GEMM)     # fp32: no SIMT path
    rc = L.flce_ce_only_from_host(ctypes.byref(pf), fake, fake, fake, fake, None, fake, 1 << 40, None, None)
    assert rc == B.FLCE_ERR_UNSUPPORTED


def test_scale_gradient_host_errors(L):
    """Argument errors come back before any device call (the pointers are never
    dereferenced), and n = 0 is a no-op."""
    from linear_cross_entropy_02_gb300 import _lib as B
    bf, f32 = B.FLCE_DTYPE_BF16, B.FLCE_DTYPE_F32
    x = ctypes.c_void_p(1 << 20)
    assert L.flce_scale_gradient(x, bf, ctypes.c_void_p(1 << 21), bf, -1, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(x, 7, ctypes.c_void_p(1 << 21), bf, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(x, bf, ctypes.c_void_p(1 << 21), -1, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(None, bf, ctypes.c_void_p(1 << 21), bf, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(x, f32, None, f32, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(None, bf, None, bf, 0, None, None) == B.FLCE_OK
    # partial overlaps, and an exact alias that changes the element size
    assert L.flce_scale_gradient(x, f32, ctypes.c_void_p((1 << 20) + 16), f32, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(ctypes.c_void_p((1 << 20) + 30), bf, x, bf, 16, None, None) == B.FLCE_ERR_ARG
    assert L.flce_scale_gradient(x, f32, x, bf, 16, None, None) == B.FLCE_ERR_ARG


def test_binding_rejects_cpu_tensors():
    import torch
    import linear_cross_entropy_02_gb300 as flce
    h = torch.zeros(4, 8, dtype=torch.bfloat16)
    W = torch.zeros(16, 8, dtype=torch.bfloat16)
    y = torch.zeros(4, dtype=torch.int64)
    with pytest.raises(ValueError, match="CUDA"):
        flce.flce_ce_only(h, W, y)


def test_params_struct_matches_header():
    """ctypes' FlceParams has the fields of the header's flce_params, in order and
    with the same C types, so the two agree on the struct's layout."""
    from linear_cross_entropy_02_gb300._lib import FlceParams
    with open(os.path.join(ROOT, "include", "flce.h")) as f:
        src = f.read()
    body = src[src.index("typedef struct flce_params {"):src.index("} flce_params;")]
    body = re.sub(r"/\*.*?\*/", "", body, flags=re.S)
    decl = re.findall(r"^\s*(int64_t|int32_t|float)\s+(\w+);", body, flags=re.M)
    ctype = {"int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32, "float": ctypes.c_float}
    assert [(n, ctype[t]) for t, n in decl] == list(FlceParams._fields_)
    assert ctypes.sizeof(FlceParams) == 104


def test_chunk_rows_for_budget(L):
    """The budget helper returns the largest 128-multiple chunk whose workspace
    fits, and smaller budgets never give larger chunks."""
    import linear_cross_entropy_02_gb300 as flce
    from linear_cross_entropy_02_gb300 import _lib as B
    N, H, V = 32768, 7168, 129280
    last = 1 << 30
    for gb in (20, 8, 4, 1):
        c = flce.flce_chunk_rows_for_budget(N, H, V, gb << 30)
        assert c % 128 == 0 and c <= last
        last = c
        if c:
            assert flce.flce_workspace_size(N, H, V, chunk_rows=c) <= gb << 30
            if c < 32768:
                assert flce.flce_workspace_size(N, H, V, chunk_rows=c + 128) > gb << 30
    # the recompute backward fits budgets the stored-logits one does not
    tiny = 64 << 20
    assert flce.flce_chunk_rows_for_budget(N, H, V, tiny) == 0
    assert flce.flce_chunk_rows_for_budget(N, H, V, tiny, flags=B.FLCE_FLAG_RECOMPUTE) > 0


def test_missing_library_fails_loudly(tmp_path):
    """Without the built library there is no fallback: the first call raises
    and names the build step (checked in a fresh interpreter that points the
    loader at a path with no library)."""
    import subprocess
    import sys
    code = (
        "import sys, torch\n"
        f"sys.path.insert(0, {ROOT!r})\n"
        "from linear_cross_entropy_02_gb300 import _lib\n"
        f"_lib.LIB_PATH = {str(tmp_path / 'absent.so')!r}\n"
        "import linear_cross_entropy_02_gb300 as flce\n"
        "try:\n"
        "    flce.flce_workspace_size(16, 64, 100)\n"
        "except RuntimeError as e:\n"
        "    print('raised:', e)\n"
        "    sys.exit(0)\n"
        "sys.exit(3)\n")
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "no CPU or PyTorch fallback" in r.stdout


def test_vocab_parallel_host_errors(L):
    """The vocab-parallel entry points reject a shard that is not inside the
    vocabulary, and shard tables that do not tile it or do not contain the
    calling shard, before any device call (the pointers are never used)."""
    from linear_cross_entropy_02_gb300 import _lib as B
    fake = ctypes.c_void_p(1 << 20)
    p = _params(L, n_rows=64, hidden=32, vocab=300)
    assert L.flce_vp_workspace_size(ctypes.byref(p), 0, 0, 0) == \
        L.flce_workspace_size(ctypes.byref(p), B.FLCE_MODE_CE_ONLY, 0, 0)
    bwd = L.flce_vp_workspace_size(ctypes.byref(p), 1, 1, 1)
    assert bwd > L.flce_vp_workspace_size(ctypes.byref(p), 1, 0, 0) >= 64 * 4
    # the shard [vocab_offset, vocab_offset + 300) must lie inside [0, vocab_total)
    for off, tot in ((0, 299), (-1, 600), (301, 600), (0, 1 << 31)):
        rc = L.flce_vp_forward(ctypes.byref(p), off, tot, fake, fake, fake, fake, fake, 1 << 40, None)
        assert rc == B.FLCE_ERR_ARG, (off, tot)
    assert L.flce_vp_forward(ctypes.byref(p), 0, 600, fake, fake, fake, None, fake, 1 << 40, None) == B.FLCE_ERR_ARG
    pf = _params(L, n_rows=64, hidden=32, vocab=300, dtype=B.FLCE_DTYPE_F32)
    assert L.flce_vp_forward(ctypes.byref(pf), 0, 600, fake, fake, fake, fake, fake, 1 << 40, None) == \
        B.FLCE_ERR_UNSUPPORTED

    def bwd_rc(offsets, off=0, tot=600, params=p, ws=1 << 40):
        arr = (ctypes.c_int64 * len(offsets))(*offsets)
        return L.flce_vp_backward(ctypes.byref(params), off, tot, len(offsets) - 1, arr, fake, fake, fake, fake,
                                  fake, None, None, None, fake, fake, fake, ws, None)
    for bad in ([0, 600], [0, 300, 599], [1, 300, 600], [0, 250, 600], [0, 300, 300, 600]):
        assert bwd_rc(bad) == B.FLCE_ERR_ARG, bad
    assert bwd_rc([0, 300, 600], ws=bwd - 256) == B.FLCE_ERR_WORKSPACE
    assert bwd_rc([0, 300, 600], params=pf) == B.FLCE_ERR_UNSUPPORTED
    assert bwd_rc(list(range(0, 600, 9)) + [600]) == B.FLCE_ERR_ARG          # 67 shards: more than 64


def test_vocab_parallel_stored_host_errors(L):
    """FLCE_FLAG_VP_STORED: one workspace size for both calls, larger than
    either call's without it (it holds the logits of every row, growing with
    N, and one chunk's dlogits); the flag is refused with the recompute or
    K-major backward, and a short workspace is refused, all before any device
    call."""
    from linear_cross_entropy_02_gb300 import _lib as B
    fake = ctypes.c_void_p(1 << 20)
    p = _params(L, n_rows=64, hidden=32, vocab=300)
    ps = _params(L, n_rows=64, hidden=32, vocab=300, flags=B.FLCE_FLAG_VP_STORED)
    fwd_s = L.flce_vp_workspace_size(ctypes.byref(ps), 0, 0, 0)
    bwd_s = L.flce_vp_workspace_size(ctypes.byref(ps), 1, 1, 1)
    assert fwd_s == bwd_s > L.flce_vp_workspace_size(ctypes.byref(p), 1, 1, 1)
    assert fwd_s > L.flce_vp_workspace_size(ctypes.byref(p), 0, 0, 0) + 64 * 300 * 4   # fp16 logits + bf16 dz
    for extra in (B.FLCE_FLAG_RECOMPUTE, B.FLCE_FLAG_KMAJOR_BWD):
        pb = _params(L, n_rows=64, hidden=32, vocab=300, flags=B.FLCE_FLAG_VP_STORED | extra)
        assert L.flce_vp_workspace_size(ctypes.byref(pb), 0, 0, 0) == 0
        assert L.flce_vp_forward(ctypes.byref(pb), 0, 600, fake, fake, fake, fake, fake, 1 << 40, None) == \
            B.FLCE_ERR_ARG
    big = [L.flce_vp_workspace_size(ctypes.byref(_params(L, n_rows=n, hidden=32, vocab=300,
                                                          flags=B.FLCE_FLAG_VP_STORED)), 0, 0, 0)
           for n in (40000, 80000)]
    assert big[1] - big[0] >= 40000 * 300 * 2                 # the kept fp16 logits grow with N
    arr = (ctypes.c_int64 * 3)(0, 300, 600)
    rc = L.flce_vp_backward(ctypes.byref(ps), 0, 600, 2, arr, fake, fake, fake, fake, fake, None, None, None, fake,
                            fake, fake, bwd_s - 256, None)
    assert rc == B.FLCE_ERR_WORKSPACE
