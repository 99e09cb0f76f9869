"""Guard bands: every output buffer (and the split-K workspace) is placed
inside a larger allocation whose margins are filled with a poison pattern;
after the call the margins must still hold it, and the interior must equal
the result of the same call into a plain buffer.  This is the stand-in for a
memory checker on the ragged edges of the three matmul kernels (last row
tile, last token tile, split tiles), of the fused gate/up layer and of the
pack (ragged N, zero-point words of a ragged group count)."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")

PAD = 4096   # elements of margin on each side
POISON = {torch.float16: 0x7E5B, torch.int32: 0x5A5A5A5B, torch.uint8: 0xA5, torch.float32: 0x7FC0DEAD}


def _banded(shape, dtype):
    n = int(np.prod(shape))
    bits = {torch.float16: torch.int16, torch.int32: torch.int32, torch.uint8: torch.uint8,
            torch.float32: torch.int32}[dtype]
    p = POISON[dtype]
    if bits == torch.int16 and p >= 1 << 15:
        p -= 1 << 16
    flat = torch.full((n + 2 * PAD,), p, dtype=bits, device="cuda")
    view = flat[PAD:PAD + n].view(dtype).view(shape)
    return view, flat, p


def _check_bands(flat, p, n):
    torch.cuda.synchronize()
    lo, hi = flat[:PAD], flat[PAD + n:]
    assert bool((lo == p).all()), "the call wrote below its buffer"
    assert bool((hi == p).all()), "the call wrote past its buffer"


def _layer(N, K, seed, w_bit=4, group=128):
    g = torch.Generator(device="cuda").manual_seed(seed)
    W = (torch.randn((N, K), generator=g, device="cuda") * 0.02).half()
    s_c = torch.rand(K, generator=g, device="cuda") * 2 + 0.25
    inv_s = 1.0 / s_c
    q, s, z = awq.pack(W, s_c, w_bit=w_bit, group=group)
    return W, s_c, inv_s, (q, s, z)


def _tokens(M, K, seed):
    g = torch.Generator(device="cuda").manual_seed(seed)
    return torch.randn((M, K), generator=g, device="cuda").half()


@pytest.mark.parametrize("M,N,K", [(1, 1096, 2304), (3, 1096, 2304), (8, 264, 11008),
                                   (2, 136, 28672), (1, 40, 1152)])
def test_gemv_bands(M, N, K):
    _, _, inv_s, (q, s, z) = _layer(N, K, N + K)
    X = _tokens(M, K, M)
    ref = awq.gemv(X, q, s, z, inv_s)
    Y, flat, p = _banded((M, N), torch.float16)
    awq.gemv(X, q, s, z, inv_s, out=Y)
    _check_bands(flat, p, M * N)
    assert torch.equal(Y, ref)


@pytest.mark.parametrize("w_bit,group", [(8, 128), (4, 64), (4, 32)])
def test_gemv_variant_bands(w_bit, group):
    M, N, K = 5, 1096, 2304
    _, _, inv_s, (q, s, z) = _layer(N, K, 3 + w_bit + group, w_bit, group)
    X = _tokens(M, K, 4)
    ref = awq.gemv(X, q, s, z, inv_s)
    Y, flat, p = _banded((M, N), torch.float16)
    awq.gemv(X, q, s, z, inv_s, out=Y)
    _check_bands(flat, p, M * N)
    assert torch.equal(Y, ref)


# M <= 8 (decode matmul), narrow-token kernel with and without split-K, wide
# kernel with a ragged token tile, plain split-K and the ragged-round split
@pytest.mark.parametrize("M,N,K", [(5, 1096, 4096), (24, 1096, 4096), (48, 640, 8192),
                                   (100, 1096, 4096), (300, 1096, 4096), (130, 1024, 4096),
                                   (300, 9736, 4096)])
def test_gemm_bands(M, N, K):
    _, _, inv_s, (q, s, z) = _layer(N, K, 7 * N + K)
    X = _tokens(M, K, M + 1)
    ref = awq.gemm(X, q, s, z, inv_s)
    Y, flat, p = _banded((M, N), torch.float16)
    nws = awq.gemm_workspace_bytes(M, N, K)
    ws, wflat, wp = _banded((nws,), torch.uint8)
    awq.gemm(X, q, s, z, inv_s, out=Y, workspace=ws)
    _check_bands(flat, p, M * N)
    _check_bands(wflat, wp, nws)
    assert torch.equal(Y, ref)


@pytest.mark.parametrize("M", [1, 4, 40, 300])
def test_silu_mul_bands(M):
    I, K = 1032, 2048
    _, _, inv_s, (q, s, z) = _layer(2 * I, K, 11 + M)
    X = _tokens(M, K, 12 + M)
    fn = awq.gemv_silu_mul if M <= 8 else awq.gemm_silu_mul
    ref = fn(X, q, s, z, inv_s)
    Y, flat, p = _banded((M, I), torch.float16)
    fn(X, q, s, z, inv_s, out=Y)
    _check_bands(flat, p, M * I)
    assert torch.equal(Y, ref)


@pytest.mark.parametrize("N,K,w_bit,group", [(1096, 2304, 4, 128), (1000, 1152, 4, 128),
                                             (520, 2304, 8, 64), (264, 1024, 4, 32)])
def test_pack_bands(N, K, w_bit, group):
    W, s_c, _, (q0, s0, z0) = _layer(N, K, N, w_bit, group)
    c = 32 // w_bit
    G = K // group
    q, fq, pq = _banded((N, K // c), torch.int32)
    s, fs, ps = _banded((N, G), torch.float16)
    z, fz, pz = _banded((N, (G + c - 1) // c), torch.int32)
    awq.pack(W, s_c, w_bit=w_bit, group=group, out=(q, s, z))
    _check_bands(fq, pq, q.numel())
    _check_bands(fs, ps, s.numel())
    _check_bands(fz, pz, z.numel())
    assert torch.equal(q, q0) and torch.equal(s, s0) and torch.equal(z, z0)
