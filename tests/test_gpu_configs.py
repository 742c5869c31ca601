"""GPU parity on the configured workloads' own shapes, against the CPU oracle.

- The untied quantized output head (K=3584, N=152064; "The 4-bit CPU path",
  section "W4A8 - _C::int4_scaled_mm_cpu": the head must be untied and
  quantized) at decode sizes on every path. Only the head's 1188 row blocks
  reach the GEMV grid without a split-K cluster and the 1188-tile persistent
  grid of 16-token e4m3 tensor-core tiles.
- The head at prefill sizes M = 2048 and 4096, including one whole 128-token
  tile (every row of the last token tile) against sampled columns.
- A reduced full-model linear pass: two layers of the seven Qwen2.5-7B-shaped
  linears, each layer with its own weight seeds, plus the head, at
  M in {1, 8, 64, 512, 4096}.
- Sibling linears sharing one input (q|k|v, gate|up) run as one launch by the
  grouped calls, on both kernel paths.

Outputs are compared with the oracle on sampled rows and columns (the first and
last 128-row weight blocks, plus seeded random columns), against the bar in
tests/helpers.py; activation codes are compared bit for bit where the test
quantizes them.
"""
import numpy as np
import pytest

import oracle
import synth
from helpers import check_bf16_output, to_dev, to_host_bits

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if not torch.cuda.is_available():  # pragma: no cover - collected on CPU, skipped there
    pytest.skip("no CUDA device", allow_module_level=True)

import w4a8_quantized_gemm_gb300 as eg  # noqa: E402

HEAD_K, HEAD_N = 3584, 152064
SHAPES_7B = [("q", 3584, 3584), ("k", 3584, 512), ("v", 3584, 512), ("o", 3584, 3584),
             ("gate", 3584, 18944), ("up", 3584, 18944), ("down", 18944, 3584)]
# which activation feeds each linear (siblings share one)
INPUT_OF = {"q": 0, "k": 0, "v": 0, "o": 3, "gate": 4, "up": 4, "down": 6, "head": 7}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    eg.load()
    torch.cuda.set_device(0)
    yield
    assert eg.device_status() == 0


def _pack(w):
    return eg.pack_w4(to_dev(w.w_q), to_dev(w.scale_f16, torch.float16), to_dev(w.zero))


def _cols(N, seed, n_random=256):
    rng = np.random.default_rng(seed)
    return np.unique(np.concatenate([np.arange(128), np.arange(N - 128, N),
                                     rng.choice(N, n_random, replace=False)]))


def _check(x, w, y_bits, rows, cols, what):
    a_q, a_s, _ = oracle.quant_act(x[rows])
    _, y_ref = oracle.w4a8(a_q, a_s, w.w_q[cols], w.scale_f16[cols], w.zero[cols])
    check_bf16_output(y_bits[np.ix_(rows, cols)], y_ref, what)


@pytest.fixture(scope="module")
def head():
    w = synth.w4_weights(3, 0, synth.LINEARS["head"], HEAD_N, HEAD_K)
    return w, _pack(w)


@pytest.mark.parametrize("path", [eg.PATH_AUTO, eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [1, 4, 8, 16, 64])
def test_head_decode_sizes(head, path, M):
    w, packed = head
    x = synth.activations(3, 0, INPUT_OF["head"], M, HEAD_K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    a_q, a_s, asum = oracle.quant_act(x)
    assert np.array_equal(a.a_q.cpu().numpy(), a_q)
    assert np.array_equal(a.a_gsum.cpu().numpy(), asum)
    y = eg.w4a8_gemm(a, packed, HEAD_N, HEAD_K, path=path)
    _check(x, w, to_host_bits(y), np.arange(M), _cols(HEAD_N, 100 + M),
           f"head M={M} path={path}")


@pytest.mark.parametrize("path", [eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [1, 16])
def test_head_decode_group_partials(head, path, M):
    """Exact integer partials of the head's first and last row blocks (the
    readout runs the same main loop over the whole head)."""
    w, packed = head
    x = synth.activations(3, 1, INPUT_OF["head"], M, HEAD_K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    Q = eg.w4a8_group_partials(a, packed, HEAD_N, HEAD_K, path=path)
    a_q, _, _ = oracle.quant_act(x)
    for blk in (slice(0, 128), slice(HEAD_N - 128, HEAD_N)):
        ref = oracle.group_partials(a_q, w.w_q[blk], w.zero[blk])
        assert np.array_equal(Q[:, blk].cpu().numpy(), ref), (path, M, blk)
    del Q


@pytest.mark.parametrize("M", [2048, 4096])
def test_head_prefill_sizes(head, M):
    w, packed = head
    x = synth.activations(3, 2, INPUT_OF["head"], M, HEAD_K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = to_host_bits(eg.w4a8_gemm(a, packed, HEAD_N, HEAD_K))
    rng = np.random.default_rng(M)
    rows = np.unique(np.concatenate([np.arange(4), np.arange(M - 4, M),
                                     rng.choice(M, 8, replace=False)]))
    _check(x, w, y, rows, _cols(HEAD_N, M), f"head M={M}")
    # one whole 128-token tile (the last) against a column sample
    tile = np.arange(M - 128, M)
    _check(x, w, y, tile, _cols(HEAD_N, M + 1, n_random=64), f"head M={M} last token tile")


@pytest.fixture(scope="module")
def two_layers():
    layers = []
    for layer in range(2):
        packs = {}
        for (nm, K, N) in SHAPES_7B:
            w = synth.w4_weights(3, layer, synth.LINEARS[nm], N, K)
            packs[nm] = (w, _pack(w))
        layers.append(packs)
    return layers


@pytest.mark.parametrize("M", [1, 8, 64, 512, 4096])
def test_reduced_model_pass(two_layers, head, M):
    """Two layers x seven linears + head at one M, AUTO path, each layer's
    weights from its own seeds and each linear input quantized once."""
    rng = np.random.default_rng(1000 + M)
    rows = np.arange(M) if M <= 8 else np.unique(np.concatenate(
        [np.arange(2), np.arange(M - 2, M), rng.choice(M, 6, replace=False)]))
    for layer, packs in enumerate(two_layers):
        acts = {}
        for (nm, K, N) in SHAPES_7B:
            inp = INPUT_OF[nm]
            if inp not in acts:
                x = synth.activations(3, layer, inp, M, K)
                acts[inp] = (x, eg.quant_act(to_dev(x, torch.bfloat16)))
            x, a = acts[inp]
            w, packed = packs[nm]
            y = eg.w4a8_gemm(a, packed, N, K)
            _check(x, w, to_host_bits(y), rows, _cols(N, layer * 10 + M, n_random=min(256, N - 256)),
                   f"layer {layer} {nm} M={M}")
    w, packed = head
    x = synth.activations(3, 5, INPUT_OF["head"], M, HEAD_K)
    y = eg.w4a8_gemm(eg.quant_act(to_dev(x, torch.bfloat16)), packed, HEAD_N, HEAD_K)
    _check(x, w, to_host_bits(y), rows, _cols(HEAD_N, 7 + M, n_random=128), f"head M={M}")


@pytest.mark.parametrize("M", [2048, 4096])
def test_down_projection_split_tail_sampled(M):
    """The down projection (K = 18944) at 2048 and 4096 tokens: 192-token tiles
    whose short last round runs as a split-K second launch. Rows from every
    region (first, last -- the last m-tile holds the split tiles on this
    grid -- and random) against sampled columns including the last 384."""
    K, N = 18944, 3584
    assert eg.tc_token_tile(M, N, K) == 192 and eg.tc_launches(M, N, K) == 2
    w = synth.w4_weights(3, 9, synth.LINEARS["down"], N, K)
    packed = _pack(w)
    x = synth.activations(3, 9, INPUT_OF["down"], M, K)
    y = to_host_bits(eg.w4a8_gemm(eg.quant_act(to_dev(x, torch.bfloat16)), packed, N, K))
    rng = np.random.default_rng(M + 7)
    rows = np.unique(np.concatenate([np.arange(2), np.arange(M - 64, M, 9),
                                     rng.choice(M, 6, replace=False)]))
    cols = np.unique(np.concatenate([_cols(N, M + 8, n_random=128), np.arange(N - 384, N)]))
    _check(x, w, y, rows, cols, f"down M={M} (split tail)")


def test_w8a8_bench_shape_sampled():
    """W8A8 at the bench's shape (4096 x 12288 x 3072, 192-token tiles) on
    sampled rows and columns against the int8-dynamic oracle."""
    M, N, K = 4096, 12288, 3072
    assert eg.tc_token_tile(M, N, K, eg.VARIANT_W8A8) == 192
    x = synth.activations(5, 2, 0, M, K)
    w8, s8 = synth.w8_weights(5, 2, 0, N, K)
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    y = to_host_bits(eg.w8a8_gemm(a, to_dev(w8), to_dev(s8, torch.float16)))
    rng = np.random.default_rng(12)
    rows = np.unique(np.concatenate([[0, 1, M - 1], rng.choice(M, 6, replace=False)]))
    cols = _cols(N, 13)
    a_q, a_s, _ = oracle.quant_act(x[rows])
    _, _, y_ref = oracle.w8a8(a_q, a_s, w8[cols], s8[cols])
    check_bf16_output(y[np.ix_(rows, cols)], y_ref, "W8A8 4096 x 12288 x 3072")


# --------------------------------------------------- sibling linears, one launch

@pytest.mark.parametrize("path", [eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [1, 3, 16, 17, 200])
def test_grouped_siblings_match_oracle(path, M):
    """Three linears of different widths (one, three and two 128-row blocks)
    sharing one input, in one launch: every output against the oracle, as is
    each linear's separate call on the same path."""
    K = 1024
    Ns = [128, 384, 256]
    x = synth.activations(11, M, 0, M, K)
    ws = [synth.w4_weights(11, 0, j, n, K) for j, n in enumerate(Ns)]
    packs = [_pack(w) for w in ws]
    a = eg.quant_act(to_dev(x, torch.bfloat16))
    ys = eg.w4a8_gemm_grouped(a, packs, Ns, K, path=path)
    a_q, a_s, _ = oracle.quant_act(x)
    for j, (w, y) in enumerate(zip(ws, ys)):
        _, y_ref = oracle.w4a8(a_q, a_s, w.w_q, w.scale_f16, w.zero)
        check_bf16_output(to_host_bits(y), y_ref, f"grouped linear {j} M={M} path={path}")
        y_sep = eg.w4a8_gemm(a, packs[j], Ns[j], K, path=path)
        check_bf16_output(to_host_bits(y_sep), y_ref, f"separate linear {j}")
    assert eg.device_status() == 0


@pytest.mark.parametrize("M", [1, 4, 16, 512])
def test_grouped_7b_siblings_sampled(M):
    """q|k|v and gate|up of one Qwen2.5-7B layer through the one-call grouped
    linear (AUTO path), sampled against the oracle."""
    for names in (["q", "k", "v"], ["gate", "up"]):
        K = 3584
        Ns = [n for (nm, _, n) in SHAPES_7B if nm in names]
        ws = [synth.w4_weights(3, 0, synth.LINEARS[nm], n, K) for nm, n in zip(names, Ns)]
        x = synth.activations(3, 0, INPUT_OF[names[0]], M, K)
        ys = eg.w4a8_linear_grouped(to_dev(x, torch.bfloat16), [_pack(w) for w in ws], Ns)
        rng = np.random.default_rng(M)
        rows = np.arange(M) if M <= 16 else np.unique(np.concatenate(
            [np.arange(2), np.arange(M - 2, M), rng.choice(M, 6, replace=False)]))
        for nm, n, w, y in zip(names, Ns, ws, ys):
            _check(x, w, to_host_bits(y), rows, _cols(n, M, n_random=min(256, n - 256)),
                   f"grouped {nm} M={M}")


@pytest.mark.parametrize("path", [eg.PATH_AUTO, eg.PATH_GEMV, eg.PATH_TC])
@pytest.mark.parametrize("M", [2, 16, 130])
def test_linear_grouped_equals_quant_then_grouped_gemm(path, M):
    K, Ns = 512, [256, 128]
    x = to_dev(synth.activations(12, 0, 0, M, K), torch.bfloat16)
    packs = [_pack(synth.w4_weights(12, 0, j, n, K)) for j, n in enumerate(Ns)]
    y1 = eg.w4a8_linear_grouped(x, packs, Ns, path=path)
    use = path if path != eg.PATH_AUTO else eg.auto_path(M)
    y2 = eg.w4a8_gemm_grouped(eg.quant_act(x), packs, Ns, K, path=use)
    for a, b in zip(y1, y2):
        assert torch.equal(a, b)


def test_grouped_refusals():
    import ctypes
    lib = eg.load()
    M, K = 4, 512
    a = eg.quant_act(to_dev(synth.activations(12, 1, 0, M, K), torch.bfloat16))
    p = _pack(synth.w4_weights(12, 1, 0, 256, K))
    y = torch.empty((M, 256), dtype=torch.bfloat16, device="cuda")
    st = torch.cuda.current_stream().cuda_stream

    def call(count, packs, Ns, ys):
        P = (ctypes.c_void_p * max(1, len(packs)))(*packs)
        Nn = (ctypes.c_int64 * max(1, len(Ns)))(*Ns)
        Y = (ctypes.c_void_p * max(1, len(ys)))(*ys)
        return lib.egopq_w4a8_gemm_grouped(a.a_q.data_ptr(), a.a_tc.data_ptr(), a.a_s.data_ptr(),
                                           a.a_gsum.data_ptr(), count, P, Nn, M, K, 128, Y, 0, st)

    ok = ([p.data_ptr()], [256], [y.data_ptr()])
    assert call(1, *ok) == 0
    assert call(0, *ok) == -1
    assert call(9, [p.data_ptr()] * 9, [256] * 9, [y.data_ptr()] * 9) == -1
    assert call(1, [p.data_ptr()], [200], [y.data_ptr()]) == -2
    assert call(1, [p.data_ptr()], [256], [y.data_ptr() + 4]) == -3
    assert call(1, [0], [256], [y.data_ptr()]) == -1
    assert eg.device_status() == 0
