"""Canary padding: every output (O, LSE, the decode workspace) sits between guard regions
filled with a sentinel byte pattern; after the call the guards must be untouched.  The shapes
are ragged (rows and keys that are not multiples of the tiles, odd head counts) so that each
path's last tile, last split and last row group write next to a guard."""
import pytest
import torch

import streaming_attention_flashattention_gb300 as gb

pytestmark = pytest.mark.gpu

GUARD = 4096            # bytes on each side; a multiple of 256, so the payload stays aligned
SENTINEL = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _built():
    from streaming_attention_flashattention_gb300 import build
    build.build()
    gb.load_library()
    yield
    st, word = gb.attn_last_device_error()
    assert st == 0 and word == 0, f"device error word set: {word}"


class Guarded:
    """A device tensor of `shape` inside [guard | payload | guard] bytes; `shift` moves the
    payload by that many bytes (to make it 16- but not 32-byte aligned)."""

    def __init__(self, shape, dtype, shift=0):
        esize = torch.empty((), dtype=dtype).element_size()
        n = 1
        for s in shape:
            n *= s
        self.nbytes = n * esize
        self.lo = GUARD + shift
        self.buf = torch.full((self.lo + self.nbytes + GUARD,), SENTINEL, dtype=torch.uint8,
                              device="cuda")
        self.t = self.buf[self.lo:self.lo + self.nbytes].view(dtype).view(shape)

    def check(self, name):
        torch.cuda.synchronize()
        head = self.buf[:self.lo]
        tail = self.buf[self.lo + self.nbytes:]
        assert bool((head == SENTINEL).all()), f"{name}: bytes written before the output"
        assert bool((tail == SENTINEL).all()), f"{name}: bytes written after the output"


def randn(shape, seed, dtype=torch.bfloat16):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(dtype).cuda()


@pytest.mark.parametrize("B,Hq,Hkv,Sq,Skv,causal,dtype,shift", [
    (1, 6, 2, 300, 777, True, torch.bfloat16, 0),         # KV-split mode, ragged rows and keys
    (1, 6, 2, 300, 777, True, torch.bfloat16, 16),        # 16-byte aligned output: 16-byte stores
    (1, 64, 8, 1300, 1300, True, torch.bfloat16, 0),      # pair mode (352 pairs), ragged last Q tile
    (1, 32, 8, 4096, 4096, False, torch.bfloat16, 0),     # pairs plus the KV-split tail launch
    (2, 3, 1, 130, 200, False, torch.float32, 0),         # fp32 path
    (1, 4, 4, 70, 70, True, torch.bfloat16, 0),           # d = 64 below
])
def test_prefill_writes_stay_inside(B, Hq, Hkv, Sq, Skv, causal, dtype, shift):
    d = 64 if (Hq, Sq) == (4, 70) else 128
    q = randn((B, Hq, Sq, d), 1, dtype)
    k = randn((B, Hkv, Skv, d), 2, dtype)
    v = randn((B, Hkv, Skv, d), 3, dtype)
    o = Guarded((B, Hq, Sq, d), dtype, shift)
    lse = Guarded((B, Hq, Sq), torch.float32)
    gb.attn_fwd(q, k, v, causal=causal, out=o.t, lse=lse.t)
    o.check("o")
    lse.check("lse")
    assert bool(torch.isfinite(o.t.float()).all())


def test_chunked_prefill_writes_stay_inside():
    B, Hq, Hkv, Sq, ctx, Lmax, d = 2, 8, 2, 200, 1300, 2048, 128
    q = randn((B, Hq, Sq, d), 4)
    kc = randn((B, Hkv, Lmax, d), 5)
    vc = randn((B, Hkv, Lmax, d), 6)
    o = Guarded((B, Hq, Sq, d), torch.bfloat16)
    lse = Guarded((B, Hq, Sq), torch.float32)
    gb.attn_prefill_kvcache(q, kc, vc, ctx, causal=True, out=o.t, lse=lse.t)
    o.check("o")
    lse.check("lse")


@pytest.mark.parametrize("B,Hq,Hkv,Tq,Lmax,lens,ns", [
    (3, 24, 3, 1, 1000, [1000, 1, 513], 5),          # warp kernel, combine
    (1, 8, 1, 1, 4096, [4001], 8),                   # warp kernel, single launch
    (3, 16, 2, 5, 3000, [3000, 7, 1500], 0),         # 40 rows per KV head: tcgen05 kernel
    (2, 8, 2, 3, 9000, [9000, 4100], 4),             # 12 rows, long splits: tcgen05, 16 Q rows loaded
    (2, 4, 2, 5, 300, [2, 300], 2),                  # 10 rows, short splits: warp kernel, two chunks
    (1, 16, 2, 20, 1300, [1300], 3),                 # 160 rows: two 128-row tiles
])
def test_decode_writes_stay_inside(B, Hq, Hkv, Tq, Lmax, lens, ns):
    d = 128
    q = randn((B, Hq, Tq, d), 7)
    kc = randn((B, Hkv, Lmax, d), 8)
    vc = randn((B, Hkv, Lmax, d), 9)
    kl = torch.tensor(lens, dtype=torch.int32, device="cuda")
    need = gb.load_library().attn_decode_multitoken_workspace_size(B, Hq, Hkv, Tq, Lmax, d, ns)
    ws = Guarded((need,), torch.uint8)
    o = Guarded((B, Hq, Tq, d), torch.bfloat16)
    lse = Guarded((B, Hq, Tq), torch.float32)
    gb.attn_decode_multitoken(q, kc, vc, kl, num_splits=ns, out=o.t, lse=lse.t, workspace=ws.t)
    o.check("o")
    lse.check("lse")
    ws.check("workspace")
    assert bool(torch.isfinite(o.t.float()).all())
