"""CPU-only checks of the C ABI: the library builds, loads, exports every
symbol declared in include/fa.h, and rejects bad arguments on the host
before touching the GPU (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "fa.h")


@pytest.fixture(scope="module")
def lib():
    from exact_attention_33_gb300.build import build
    path = build()
    import exact_attention_33_gb300 as fa
    assert os.path.samefile(path, fa.library_path())
    return fa.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


# The exported calls, exactly: the three calls of the statement of the
# problem (dense, packed varlen and paged decode with its workspace size and
# per-call status), the further prefill layouts and the backward pass, the
# allocation-free decode, and the status, self-test and version helpers.
BOUNDARY = sorted([
    "fa_fwd", "fa_fwd_varlen", "fa_decode_workspace_size", "fa_decode_paged",
    "fa_last_device_status", "fa_status_string",
    "fa_fwd_splitkv", "fa_fwd_splitkv_workspace_size", "fa_fwd_paged", "fa_fwd_fp8",
    "fa_fwd_varlen_fp8",
    "fa_bwd", "fa_bwd_varlen", "fa_bwd_workspace_size", "fa_decode_paged_noalloc",
    "fa_device_status", "fa_selftest_wait_timeout", "fa_version",
])


def test_header_declares_the_boundary():
    assert declared_functions() == BOUNDARY


def test_binding_exposes_the_boundary():
    import exact_attention_33_gb300 as fa
    for name in BOUNDARY:
        assert callable(getattr(fa, name)), name


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in fa.h but not exported"


def test_status_strings(lib):
    import exact_attention_33_gb300 as fa
    assert fa.fa_status_string(0) == "ok"
    for s in (-1, -2, -3, -4):
        assert fa.fa_status_string(s) not in ("ok", "unknown status")
    assert fa.fa_version() >= 100


P = ctypes.c_void_p(0x10000)   # never dereferenced: validation fails first
P_BAD = ctypes.c_void_p(0x10008)
NULL = ctypes.c_void_p(0)


def fwd(lib, q=P, k=P, v=P, out=P, lse=NULL, B=1, H=2, Hkv=2, N=16, d=64, scale=0.125,
        causal=0):
    return lib.fa_fwd(q, k, v, out, lse, B, H, Hkv, N, d, scale, causal, NULL)


def test_fwd_host_validation(lib):
    assert fwd(lib, q=NULL) == -1
    assert fwd(lib, k=P_BAD) == -1           # not 16-byte aligned
    assert fwd(lib, H=3, Hkv=2) == -1         # H % Hkv != 0
    assert fwd(lib, causal=2) == -1
    assert fwd(lib, scale=float("nan")) == -1
    assert fwd(lib, scale=-1.0) == -1
    assert fwd(lib, d=96) == -2
    assert fwd(lib, d=256) == -2
    assert fwd(lib, B=0) == 0                 # empty problem: no launch, success
    assert fwd(lib, N=0) == 0


def test_varlen_host_validation(lib):
    f = lib.fa_fwd_varlen
    assert f(P, P, P, P, NULL, NULL, 2, 10, 5, 2, 2, 64, 0.1, 0, NULL) == -1   # no cu_seqlens
    assert f(P, P, P, P, NULL, P, -1, 10, 5, 2, 2, 64, 0.1, 0, NULL) == -1
    assert f(P, P, P, P, NULL, P, 2, 10, 5, 2, 2, 80, 0.1, 0, NULL) == -2
    assert f(P, P, P, P, NULL, P, 0, 10, 5, 2, 2, 64, 0.1, 0, NULL) == 0


def test_decode_host_validation(lib):
    f = lib.fa_decode_paged
    base = dict(max_blocks=4, max_ctx=64, batch=2, H=8, Hkv=2, d=128, bs=16, nb=8)

    def call(ws=P, ws_bytes=1 << 20, **kw):
        a = dict(base, **kw)
        return f(P, P, P, P, a["max_blocks"], P, a["max_ctx"], a["batch"], a["H"], a["Hkv"],
                 a["d"], a["bs"], a["nb"], 0.1, P, NULL, ws, ws_bytes, NULL)
    assert call(bs=32) == -2                  # only 16-token blocks are built
    assert call(H=64, Hkv=2) == -2            # group of 32 query heads per KV head
    assert call(max_ctx=65) == -1             # table cannot hold that many tokens
    assert call(H=7) == -1
    assert call(batch=0) == 0
    assert call(ws=NULL) == -4
    assert call(ws_bytes=16) == -4
    assert call(ws=ctypes.c_void_p(0x10010)) == -4   # not 256-byte aligned


def test_workspace_size(lib):
    import exact_attention_33_gb300 as fa
    n = fa.fa_decode_workspace_size(64, 32, 8, 128, 32768, 16)
    assert n >= fa.FA_WORKSPACE_HEADER_BYTES + 64 * 32 * 128 * 4 and n % 256 == 0
    # the control block comes first in every decode and split-KV workspace
    assert fa.fa_decode_workspace_size(1, 4, 4, 64, 16, 16) > fa.FA_WORKSPACE_HEADER_BYTES
    assert fa.fa_fwd_splitkv_workspace_size(1, 4, 1024, 64, 2) > fa.FA_WORKSPACE_HEADER_BYTES
    # context lengths whose split arithmetic would leave int are refused
    assert fa.fa_decode_workspace_size(1, 32, 8, 128, 2**31 - 1, 16) == 0
    assert fa.fa_decode_workspace_size(1, 32, 8, 128, 1024, 32) == 0
    assert fa.fa_decode_workspace_size(1, 30, 8, 128, 1024, 16) == 0


def test_bwd_host_validation(lib):
    import exact_attention_33_gb300  # noqa: F401  (sets argtypes)
    f = lib.fa_bwd

    def call(q=P, lse=P, ws=P, ws_bytes=1 << 30, B=1, H=4, Hkv=2, N=300, d=128, causal=1,
             scale=0.1):
        return f(q, P, P, P, lse, P, P, P, P, B, H, Hkv, N, d, scale, causal, ws, ws_bytes, NULL)
    assert call(q=NULL) == -1
    assert call(lse=NULL) == -1
    assert call(q=P_BAD) == -1
    assert call(H=3) == -1
    assert call(causal=5) == -1
    assert call(scale=0.0) == -1
    assert call(d=96) == -2
    assert call(B=0) == 0
    assert call(N=0) == 0
    assert call(ws=NULL) == -4
    assert call(ws_bytes=16) == -4
    assert call(ws=ctypes.c_void_p(0x10010)) == -4   # not 256-byte aligned


def test_bwd_varlen_host_validation(lib):
    import exact_attention_33_gb300  # noqa: F401  (sets argtypes)
    f = lib.fa_bwd_varlen

    def call(q=P, lse=P, cu=P, ws=P, ws_bytes=1 << 30, S=3, T=500, max_len=300, H=4, Hkv=2,
             d=128, causal=1, scale=0.1):
        return f(q, P, P, P, lse, P, P, P, P, cu, S, T, max_len, H, Hkv, d, scale, causal, ws,
                 ws_bytes, NULL)
    assert call(q=NULL) == -1
    assert call(lse=NULL) == -1
    assert call(cu=NULL) == -1
    assert call(q=P_BAD) == -1
    assert call(cu=ctypes.c_void_p(0x10002)) == -1   # cu_seqlens not 4-byte aligned
    assert call(S=-1) == -1
    assert call(T=-1) == -1
    assert call(max_len=-1) == -1
    assert call(H=3) == -1
    assert call(causal=5) == -1
    assert call(scale=float("nan")) == -1
    assert call(d=96) == -2
    assert call(S=0) == 0
    assert call(T=0) == 0
    assert call(max_len=0) == 0
    assert call(ws=NULL) == -4
    assert call(ws_bytes=16) == -4
    assert call(ws=ctypes.c_void_p(0x10010)) == -4   # not 256-byte aligned


def test_bwd_workspace_size():
    import exact_attention_33_gb300 as fa
    # -lse2 and -D vectors per (batch, head), N padded to 128, then 256 bytes of
    # work counters
    assert fa.fa_bwd_workspace_size(2, 32, 8192) == 2 * 2 * 32 * 8192 * 4 + 256
    assert fa.fa_bwd_workspace_size(1, 1, 1) == 2 * 128 * 4 + 256
    assert fa.fa_bwd_workspace_size(1, 4, 129) == 2 * 4 * 256 * 4 + 256
    assert fa.fa_bwd_workspace_size(0, 4, 129) == 0


def test_fp8_host_validation(lib):
    import exact_attention_33_gb300  # noqa: F401
    f = lib.fa_fwd_fp8

    def call(q=P, B=1, H=2, Hkv=1, N=64, d=128, descales=(1.0, 1.0, 1.0), causal=0):
        return f(q, P, P, P, NULL, B, H, Hkv, N, d, 0.1, *descales, causal, NULL)
    assert call(q=NULL) == -1
    assert call(descales=(1.0, float("inf"), 1.0)) == -1
    assert call(descales=(1.0, 1.0, -2.0)) == -1
    assert call(d=96) == -2
    assert call(H=3, Hkv=2) == -1
    assert call(N=0) == 0


def test_varlen_fp8_host_validation(lib):
    import exact_attention_33_gb300  # noqa: F401  (sets argtypes)
    f = lib.fa_fwd_varlen_fp8

    def call(q=P, cu=P, n=2, T=10, mx=5, H=2, Hkv=1, d=128, descales=(1.0, 1.0, 1.0), causal=1):
        return f(q, P, P, P, NULL, cu, n, T, mx, H, Hkv, d, 0.1, *descales, causal, NULL)
    assert call(q=NULL) == -1
    assert call(cu=NULL) == -1
    assert call(descales=(1.0, float("nan"), 1.0)) == -1
    assert call(H=3, Hkv=2) == -1
    assert call(d=96) == -2
    assert call(n=0) == 0


def test_last_device_status_host_validation(lib):
    import exact_attention_33_gb300  # noqa: F401  (sets argtypes)
    assert lib.fa_last_device_status(NULL) == -1
    assert lib.fa_last_device_status(ctypes.c_void_p(0x10010)) == -1   # not 256-byte aligned


def test_workspace_header_matches_the_binding():
    import exact_attention_33_gb300 as fa
    m = re.search(r"#define\s+FA_WORKSPACE_HEADER_BYTES\s+(\d+)u", open(HEADER).read())
    assert m and int(m.group(1)) == fa.FA_WORKSPACE_HEADER_BYTES


def test_status_bits_match_the_binding():
    """The FA_DEV_* bits of include/fa.h and the binding's constants agree."""
    import exact_attention_33_gb300 as fa
    text = open(HEADER).read()
    bits = dict((name, int(val)) for name, val in
                re.findall(r"#define\s+(FA_DEV_[A-Z_]+)\s+(\d+)u", text))
    assert set(bits) == {"FA_DEV_TIMEOUT", "FA_DEV_BAD_BLOCK", "FA_DEV_BAD_CTX",
                         "FA_DEV_BAD_SEQLEN", "FA_DEV_BAD_INDEX", "FA_DEV_SMEM_ALIGN"}
    for name, val in bits.items():
        assert getattr(fa, name) == val, name
    assert len(set(bits.values())) == len(bits)
    assert all(v & (v - 1) == 0 for v in bits.values())   # one bit each


def test_binding_rejects_host_tensors_before_any_call():
    """Tensors in host memory are refused by the binding itself (no launch,
    no device pointer taken)."""
    torch = pytest.importorskip("torch")
    import exact_attention_33_gb300 as fa
    q = torch.zeros((1, 8, 2, 64), dtype=torch.bfloat16)
    for call in (lambda: fa.fa_fwd(q, q, q),
                 lambda: fa.fa_fwd_splitkv(q, q, q),
                 lambda: fa.fa_bwd(q, q, q, q, torch.zeros(1, 2, 8), q),
                 lambda: fa.fa_fwd_varlen(q[0], q[0], q[0],
                                          torch.tensor([0, 8], dtype=torch.int32), 8),
                 lambda: fa.fa_decode_paged(q[0], q, q, torch.zeros((8, 1), dtype=torch.int32),
                                            torch.ones(8, dtype=torch.int32), 1)):
        with pytest.raises(ValueError):
            call()


def test_profile_hash_covers_every_kernel_source():
    """bench.py uses a committed ncu traffic figure only while the hash of the
    kernel's sources matches the one in the summary; that hash must cover
    every local header the kernel file includes, directly or through another
    header."""
    import sys
    sys.path.insert(0, ROOT)
    import bench
    csrc = os.path.join(ROOT, "exact_attention_33_gb300", "csrc")

    def closure(name, seen):
        if name in seen:
            return seen
        seen.add(name)
        for inc in re.findall(r'#include\s+"([^"]+)"', open(os.path.join(csrc, name)).read()):
            if os.path.exists(os.path.join(csrc, inc)):
                closure(inc, seen)
        return seen

    # The public header gives the kernels only the FA_DEV_* bit values, which
    # test_status_bits_match_the_binding pins; its prose may change freely.
    public = {"../../include/fa.h"}
    for kind, main in (("prefill", "prefill.cu"), ("decode", "decode.cu")):
        listed = {os.path.basename(p) for p in bench.KERNEL_SOURCES[kind]}
        missing = closure(main, set()) - listed - public
        assert not missing, f"{kind} hash misses {sorted(missing)}"
