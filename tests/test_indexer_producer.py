"""The tensor-core indexer-logits producer: oracle pins on the CPU and GPU
parity through the C ABI."""
import numpy as np
import pytest

import workloads as wk
from oracle import default as oracle_default


@pytest.fixture(scope="module")
def orc():
    return oracle_default()


def test_e4m3_decoding_matches_torch(orc):
    torch = pytest.importorskip("torch")
    if not hasattr(torch, "float8_e4m3fn"):
        pytest.skip("torch without float8_e4m3fn")
    b = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = np.array([orc.e4m3(i) for i in range(256)])
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan) and nan.sum() == 2  # 0x7F and 0xFF
    assert np.array_equal(got[~nan], ref[~nan])
    assert np.array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def _decode(orc, b):
    table = np.array([orc.e4m3(i) for i in range(256)])
    return table[b]


def test_one_head_positive_is_a_matmul(orc):
    rng = np.random.default_rng(0)
    T, S, D = 3, 40, 128
    # positive e4m3 bytes only: every dot product is positive, ReLU is the identity
    q = rng.integers(0x18, 0x50, size=(T, 1, D)).astype(np.uint8)
    k = rng.integers(0x18, 0x50, size=(S, D)).astype(np.uint8)
    out = np.zeros((T, S), dtype=np.float32)
    orc.indexer_logits(q, k, np.ones(S, np.float32), np.ones((T, 1), np.float32), None,
                       np.full(T, S, np.int32), out)
    want = (_decode(orc, q[:, 0, :]) @ _decode(orc, k).T).astype(np.float32)
    assert np.array_equal(out, want)


def test_relu_weights_scales_and_span(orc):
    q = np.zeros((1, 2, 128), dtype=np.uint8)
    k = np.zeros((3, 128), dtype=np.uint8)
    q[0, 0, 0] = 0x38    # head 0: +1 on dim 0
    q[0, 1, 0] = 0xB8    # head 1: -1 on dim 0
    k[:, 0] = [0x40, 0xC0, 0x38]   # keys: +2, -2, +1 on dim 0
    w = np.array([[0.5, 3.0]], dtype=np.float32)
    ks = np.array([1.0, 2.0, 4.0], dtype=np.float32)
    out = np.full((1, 3), 7.0, dtype=np.float32)
    orc.indexer_logits(q, k, ks, w, [1], [3], out)
    # key 0 is before the start: untouched; key 1: head 0 dot -2 -> 0, head 1 dot +2
    # -> 3 * 2 = 6, times scale 2 -> 12; key 2: head 0 dot 1 -> 0.5, head 1 dot -1 -> 0,
    # times scale 4 -> 2
    assert out.tolist() == [[7.0, 12.0, 2.0]]


def _gpu_case(T, S, seed, starts=None, ends=None, ld_pad=0):
    torch = pytest.importorskip("torch")
    import sparse_attention_indexer_live_gb300 as dsa
    q, k, ks, w, st, en = wk.indexer_inputs(T, S, seed)
    if ends is not None:
        en = np.asarray(ends, np.int32)
    if starts is not None:
        st = np.asarray(starts, np.int32)
    dev = "cuda:0"
    out = torch.full((T, S + ld_pad), 1.5, dtype=torch.float32, device=dev)
    dsa.dsa_indexer_logits(torch.from_numpy(q).to(dev), torch.from_numpy(k).to(dev),
                           torch.from_numpy(ks).to(dev), torch.from_numpy(w).to(dev),
                           None if st is None else torch.from_numpy(st).to(dev),
                           torch.from_numpy(en).to(dev), out)
    torch.cuda.synchronize()
    assert dsa.dsa_indexer_status() == dsa.DSA_OK
    return q, k, ks, w, st, en, out.cpu().numpy()


def _check(orc, q, k, ks, w, st, en, got):
    T, S = q.shape[0], k.shape[0]
    want = np.full(got.shape, 1.5, dtype=np.float32)
    orc.indexer_logits(q, k, ks, w, st, en, want)
    # error bound of fp32 accumulation (128-term dot products on the tensor cores,
    # then a 64-term FMA chain over the heads): well under 2^-16 of the sum of
    # absolute terms; the untouched columns must be bit-identical
    tq = np.abs(_decode(orc, q))
    tk = np.abs(_decode(orc, k))
    scale = np.stack([np.abs(w[t]).astype(np.float64) @ (tq[t] @ tk.T) for t in range(T)])
    scale = scale * ks[None, :]
    live = np.zeros(got.shape, dtype=bool)
    for t in range(T):
        s0 = 0 if st is None else max(int(st[t]), 0)
        live[t, s0:min(int(en[t]), S)] = True
    assert np.array_equal(got[~live].view(np.uint32), want[~live].view(np.uint32))
    err = np.abs(got[:, :S].astype(np.float64) - want[:, :S])[live[:, :S]]
    bound = scale[live[:, :S]] * 2.0 ** -16 + 1e-30
    ratio = float((err / bound).max()) if err.size else 0.0
    assert ratio <= 1.0, f"max error / bound = {ratio}"
    return ratio


@pytest.mark.gpu
@pytest.mark.parametrize("T,S", [(4, 128), (8, 1000), (13, 4097), (64, 20_000)])
def test_gpu_producer_matches_oracle(orc, T, S):
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    got = _gpu_case(T, S, seed=T + S)
    _check(orc, *got)


@pytest.mark.gpu
def test_gpu_producer_ragged_spans():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    orc = oracle_default()
    T, S = 9, 3000
    starts = [0, 5, 129, 0, 2999, 100, 0, 1, 7]
    ends = [3000, 6, 1000, 0, 3000, 5000, 128, 2, 2048]
    got = _gpu_case(T, S, seed=3, starts=starts, ends=ends, ld_pad=37)
    _check(orc, *got)
