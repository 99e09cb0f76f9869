"""GPU parity of the decode matmul for the default format (4-bit codes,
128-channel groups, K % 256 == 0): TMA-streamed weights, warp-level MMA.

Every element of Y is checked against the oracle's fp64 linear layer within
4e-3 * sum_k |x~ w^| + 1 fp16 ulp.  The shapes reach the kernel's edge cases:
CTAs with fewer than 16 rows (the last 16-row tile reaches back into the
previous range, or below row 0), ranges that are not multiples of 16, a last
stage of 256 channels, K split over a thread-block cluster, every M from 1
to 8, with and without the channel scales.  Chains of dependent calls check
that reading the weights before the dependency wait never lets a call read
its activations early.
"""
import numpy as np
import pytest

import awq_inputs
import oracle as O

pytestmark = pytest.mark.gpu
torch = pytest.importorskip("torch")
awq = pytest.importorskip("weight_only_bit_05_b300")
from gpu_helpers import assert_linear_close, dev, host  # noqa: E402


def _layer(N, K, seed):
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
    a = np.abs(rng.standard_normal(K)).astype(np.float32) + 0.05
    s_c, inv_s = O.channel_scales(a, 0.5)
    qw, sc, zs = O.awq_pack(W, s_c)
    return qw, sc, zs, inv_s


def _tokens(M, K, seed):
    return awq_inputs.timed_tokens(M, K, 900 + seed)


SHAPES = [(8, 256), (16, 256), (24, 768), (40, 1024), (136, 2304), (264, 4352),
          (1096, 512), (520, 11008), (2200, 1280)]


@pytest.mark.parametrize("N,K", SHAPES)
@pytest.mark.parametrize("M", [1, 2, 3, 4, 5, 6, 7, 8])
def test_gemv_edges(M, N, K):
    qw, sc, zs, inv_s = _layer(N, K, N * 7 + K)
    X = _tokens(M, K, M)
    y = host(awq.gemv(dev(X), dev(qw), dev(sc), dev(zs), dev(inv_s)))
    assert_linear_close(y, X, qw, sc, zs, inv_s)


@pytest.mark.parametrize("M,N,K", [(1, 136, 28672), (2, 264, 11008), (8, 264, 4096),
                                   (8, 520, 11008), (5, 40, 8192)])
def test_gemv_cluster_split(M, N, K):
    """Activations too large for one CTA's shared memory: K slices of a
    cluster, added in rank order."""
    qw, sc, zs, inv_s = _layer(N, K, 31 + M)
    X = _tokens(M, K, 40 + M)
    y = host(awq.gemv(dev(X), dev(qw), dev(sc), dev(zs), dev(inv_s)))
    assert_linear_close(y, X, qw, sc, zs, inv_s)


def test_gemv_without_channel_scales():
    qw, sc, zs, _ = _layer(264, 2304, 5)
    X = _tokens(3, 2304, 6)
    y = host(awq.gemv(dev(X), dev(qw), dev(sc), dev(zs), None))
    assert_linear_close(y, X, qw, sc, zs, None)


def test_gemv_deterministic():
    qw, sc, zs, inv_s = _layer(2200, 4352, 9)
    X = dev(_tokens(4, 4352, 10))
    args = (dev(qw), dev(sc), dev(zs), dev(inv_s))
    y0 = awq.gemv(X, *args)
    for _ in range(3):
        assert torch.equal(awq.gemv(X, *args), y0)


def test_gemv_dependent_chain_in_graph():
    """y_{i+1} = gemv(y_i) through five layers (each call's input is the
    previous call's output), captured in a CUDA graph and replayed: the
    result must equal the same chain run call by call with a device
    synchronization in between, and the oracle's chain."""
    K = 1024
    layers = [_layer(K, K, 50 + i) for i in range(5)]
    gl = [tuple(dev(t) for t in L) for L in layers]
    X = _tokens(2, K, 60)
    gX = dev(X)
    ys = [torch.empty((2, K), dtype=torch.float16, device="cuda") for _ in layers]

    def chain():
        src = gX
        for (q, s, z, i), y in zip(gl, ys):
            awq.gemv(src, q, s, z, i, out=y)
            src = y

    ref = []
    src = gX
    for (q, s, z, i) in gl:
        src = awq.gemv(src, q, s, z, i)
        torch.cuda.synchronize()
        ref.append(src.clone())
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        chain()
    torch.cuda.current_stream().wait_stream(st)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        chain()
    for _ in range(3):
        for y in ys:
            y.zero_()
        g.replay()
        torch.cuda.synchronize()
        for y, r in zip(ys, ref):
            assert torch.equal(y, r)
    # the oracle's chain, each layer from the GPU's previous (fp16) output
    src = X
    for (qw, sc, zs, inv_s), r in zip(layers, ref):
        assert_linear_close(host(r), src, qw, sc, zs, inv_s)
        src = host(r)


def test_gemv_right_after_pack():
    """awq_pack writes the weights, awq_gemv (which reads them before its
    dependency wait) follows at once on the same stream, repeatedly with new
    weights in the same buffers."""
    N, K = 1096, 2304
    rng = np.random.default_rng(3)
    qw = torch.empty((N, K // 8), dtype=torch.int32, device="cuda")
    sc = torch.empty((N, K // 128), dtype=torch.float16, device="cuda")
    zs = torch.empty((N, (K // 128 + 7) // 8), dtype=torch.int32, device="cuda")
    X = _tokens(1, K, 70)
    gX = dev(X)
    for it in range(4):
        W = (rng.standard_normal((N, K)) * 0.02).astype(np.float16)
        gW = dev(W)
        awq.pack(gW, None, out=(qw, sc, zs))
        y = host(awq.gemv(gX, qw, sc, zs, None))
        rq, rs, rz = O.awq_pack(W, None)
        assert np.array_equal(host(qw), rq)
        assert_linear_close(y, X, rq, rs, rz, None)


# plans on 148 SMs: 16 warps with K halved over a cluster of two and 1-deep
# rings (8, 520, 11008), (7, 264, 16384); 2-deep rings (8, 1096, 8192),
# (3, 136, 28672); 16 warps without a split (5, 264, 8192)
@pytest.mark.parametrize("M,N,K", [(8, 520, 11008), (7, 264, 16384), (8, 1096, 8192),
                                   (3, 136, 28672), (5, 264, 8192)])
def test_gemm_routes_cluster_plans(M, N, K):
    """awq_gemm at up to 8 tokens runs the decode matmul also when it halves K
    over a cluster of two (with 2- or 1-deep rings): per element against the
    oracle, and the same bits as awq_gemv for the same call."""
    qw, sc, zs, inv_s = _layer(N, K, 77 + M)
    X = _tokens(M, K, 80 + M)
    args = (dev(X), dev(qw), dev(sc), dev(zs), dev(inv_s))
    y = awq.gemm(*args)
    assert torch.equal(y, awq.gemv(*args))
    assert_linear_close(host(y), X, qw, sc, zs, inv_s)
