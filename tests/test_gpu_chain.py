"""The conv chain (conv_fused_chain_*): a sequence of conv runs in one persistent launch.

Independent steps (no step reads another's output) must give, element by element, what each
conv gives on its own: the oracle within the single-conv bound.

Dependent steps are checked twice.  (1) An integer chain: integer inputs, sparse weights in
{-1, 0, 1}, no BN, a Clip(-64, 64) activation and integer residuals.  Every sum is then an
integer below 2^24 (exact in the fp32 accumulator) and every stored value an integer of
magnitude at most 64 (exact in bf16), so the kernel's chain and the oracle's are the same
numbers and must agree bit for bit; a tile that read its input, or a residual, before the step
producing it had stored it cannot pass.  (2) Bottleneck chains with He-normal weights, folded BN
and ReLU, whose intermediate outputs are rounded to bf16 on both sides (the oracle rounds its
fp64 result to float32 and then to nearest-even bf16, as the kernel rounds its fp32 result).
Where the fp32 and fp64 sums of a layer fall on opposite sides of a rounding midpoint the two
chains store values one bf16 unit apart; the next layer's sums then differ by the weights times
those units, at most a few units of bf16 rounding of that layer's largest value.  The bound
for the bottleneck chains is two units in the last place of the reference plus 2^-6 times the
step's largest output.  (The share of elements more than one unit apart is reported, not bounded:
it grows with every layer the differences pass through, from about 1% after seven layers of
512-channel bottlenecks to several percent deep in ResNet-50, while the largest difference stays
a fraction of the bound.)  The
intermediate buffers are filled with NaN before every run, so a read of a tile that was never
stored shows up as NaN.  Runs must also be bitwise repeatable (plain and graph replays), since
the arithmetic of a tile never depends on timing.
"""
import numpy as np
import pytest
import torch

import convolution_onnx_conv_gb300 as cf
from convolution_onnx_conv_gb300 import synthetic, workloads
from convolution_onnx_conv_gb300.workloads import ConvSpec, ACT_NONE, ACT_RELU, ACT_RELU6

from parity import compare, inputs_for, to_device_nhwc

import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cf.load_library(build_if_missing=True)


def S(name, N, C, H, W, K, R, S_, stride=(1, 1), pads=(0, 0, 0, 0), act=ACT_RELU, dilation=(1, 1)):
    return ConvSpec(name, N, C, H, W, K, R, S_, stride, pads, dilation, act=act, has_bn=True)


def variant_for(spec):
    plain_1x1 = spec.R == 1 and spec.S == 1 and tuple(spec.stride) == (1, 1) and tuple(spec.pads) == (0, 0, 0, 0)
    return cf.CONVF_VARIANT_GEMM_1X1 if plain_1x1 else cf.CONVF_VARIANT_IMPLICIT_GEMM


def make(spec, inp, out_bf16=False, residual=False, **kw):
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"], scale, shift,
                        stride=spec.stride, pads=spec.pads, dilation=spec.dilation, act=spec.act,
                        variant=variant_for(spec), out_bf16=out_bf16, residual=residual, **kw)


def oracle_step(spec, x, inp, residual=None):
    bn = tuple(t.numpy() for t in inp["bn"])
    return oracle.conv_bn_act(x, inp["w"].double().numpy(), None, bn, spec.act, 0.0, 6.0, spec.stride, spec.pads,
                              spec.dilation, spec.group, residual=residual)


def ulp_bf16(v):
    a = np.maximum(np.abs(np.asarray(v, dtype=np.float64)), 2.0 ** -126)
    return np.exp2(np.floor(np.log2(a)) - 7)


def chain_close(got, ref):
    """The bottleneck-chain bound (module docstring): (ok, worst ratio, fraction > 1 unit)."""
    d = np.abs(np.asarray(got, dtype=np.float64) - ref)
    u = ulp_bf16(ref)
    allow = 2 * u + 2.0 ** -6 * np.abs(ref).max()
    worst = float((d / allow).max())
    frac = float(np.mean(d > u))
    return worst <= 1.0, worst, frac


# ------------------------------------------------------------------ independent steps, fp32 out
# every activation-load form (3-D box pairs, 2-D boxes with an odd block count and a channel
# tail, im2col with strides, dilation and a 7x7 filter), both tile widths, ragged rows and
# channel blocks, and one step with more tiles than there are SMs
INDEP = [
    S("c1x1_a3d_k136", 2, 128, 20, 20, 136, 1, 1),
    S("c1x1_odd_kb_k64", 2, 192, 14, 13, 64, 1, 1, act=ACT_NONE),
    S("c1x1_c40_k96", 3, 40, 11, 9, 96, 1, 1, act=ACT_RELU6),
    S("c3x3_k72", 2, 64, 17, 19, 72, 3, 3, pads=(1, 1, 1, 1)),
    S("c3x3_s2", 3, 128, 15, 15, 128, 3, 3, (2, 2), (1, 1, 1, 1)),
    S("c1x1_s2", 2, 64, 16, 16, 128, 1, 1, (2, 2)),
    S("c3x3_dil2", 2, 64, 13, 12, 64, 3, 3, pads=(2, 2, 2, 2), dilation=(2, 2)),
    S("c7x7_s2_c16", 2, 16, 23, 22, 64, 7, 7, (2, 2), (3, 3, 3, 3)),
    S("c1x1_many_tiles", 4, 64, 56, 57, 256, 1, 1),
]


@pytest.mark.parametrize("pairs", [1, 2], ids=["single", "pairs"])
def test_independent_steps_match_the_oracle_every_output(pairs):
    steps, refs, convs, ys, keep = [], [], [], [], []
    for i, spec in enumerate(INDEP):
        inp = inputs_for(spec, 9100 + i)
        conv = make(spec, inp)
        x = to_device_nhwc(inp["x"])
        y = conv.new_output()
        steps.append((conv, x, y))
        convs.append(conv)
        ys.append(y)
        keep.append(x)
        refs.append(oracle_step(spec, inp["x"].double().numpy(), inp))
    chain = cf.ConvChain(steps, cta_pairs=pairs)
    d = chain.describe()
    assert f"steps={len(INDEP)}" in d and "out=f32" in d and f"cta_pairs={pairs - 1}" in d, d
    assert " a3d" in d and "src=-1" in d and "src=0" not in d, d
    first = None
    for run in range(3):
        for y in ys:
            y.fill_(float("nan"))
        chain()
        torch.cuda.synchronize()
        assert chain.status() == cf.CONVF_OK
        outs = [y.cpu().contiguous().numpy() for y in ys]
        for spec, got, ref in zip(INDEP, outs, refs):
            ok, worst, idx = compare(got, ref, False)
            assert ok, (spec.name, run, worst, idx)
        if first is None:
            first = outs
        else:
            assert all(np.array_equal(a, b) for a, b in zip(first, outs))
    chain.close()
    for c in convs:
        c.close()


# ------------------------------------------------------------------ dependent steps, bf16 out

def bottleneck_chain(N, H, W, cin, mid, cout, stride, blocks, seed):
    """Specs and inputs of `blocks` ResNet bottleneck blocks: the first with a 1x1 projection
    shortcut (stride `stride` on the projection and the 3x3), the others identity shortcuts.
    Each entry: (spec, inputs, source of x, source of the residual), sources being step indices
    or -1 for the chain input."""
    out = []
    h, w, c, block_in = H, W, cin, -1
    for b in range(blocks):
        st = stride if b == 0 else 1
        ho, wo = (h - 1) // st + 1, (w - 1) // st + 1
        if b == 0:
            out.append((S(f"b{b}_proj", N, c, h, w, cout, 1, 1, (st, st), act=ACT_NONE), block_in, None))
            shortcut = len(out) - 1
        else:
            shortcut = block_in
        out.append((S(f"b{b}_1x1a", N, c, h, w, mid, 1, 1), block_in, None))
        out.append((S(f"b{b}_3x3", N, mid, h, w, mid, 3, 3, (st, st), (1, 1, 1, 1)), len(out) - 1, None))
        out.append((S(f"b{b}_1x1b", N, mid, ho, wo, cout, 1, 1), len(out) - 1, shortcut))
        block_in = len(out) - 1
        h, w, c = ho, wo, cout
    return [(spec, inputs_for(spec, seed + i), src, rsrc) for i, (spec, src, rsrc) in enumerate(out)]


def run_bf16_chain(N, H, W, cin, mid, cout, stride, blocks, seed, graph=False, pairs=0):
    plan = bottleneck_chain(N, H, W, cin, mid, cout, stride, blocks, seed)
    g = torch.Generator().manual_seed(seed - 1)
    x0 = torch.randn((N, cin, H, W), generator=g).to(torch.bfloat16)
    x0d = to_device_nhwc(x0)
    convs, ys, steps = [], [], []
    for spec, inp, src, rsrc in plan:
        conv = make(spec, inp, out_bf16=True, residual=rsrc is not None)
        y = conv.new_output()
        x = x0d if src < 0 else ys[src]
        if rsrc is None:
            steps.append((conv, x, y))
        else:
            steps.append((conv, x, y, x0d if rsrc < 0 else ys[rsrc]))
        convs.append(conv)
        ys.append(y)
    chain = cf.ConvChain(steps, cta_pairs=pairs)
    # the oracle's chain: each output rounded like the kernel's (float32, then bf16)
    refs = []
    for spec, inp, src, rsrc in plan:
        x = x0.double().numpy() if src < 0 else refs[src]
        r = None if rsrc is None else (x0.double().numpy() if rsrc < 0 else refs[rsrc])
        refs.append(oracle.round_bf16(oracle_step(spec, x, inp, residual=r)))
    results = []
    if graph:
        gr = torch.cuda.CUDAGraph()
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            chain()   # warm-up outside the capture
            torch.cuda.synchronize()
            with torch.cuda.graph(gr, stream=s):
                chain()
    for run in range(3):
        for y in ys:
            y.fill_(float("nan"))
        if graph:
            gr.replay()
        else:
            chain()
        torch.cuda.synchronize()
        assert chain.status() == cf.CONVF_OK
        results.append([y.cpu().float().contiguous().numpy() for y in ys])
    d = chain.describe()
    chain.close()
    for c in convs:
        c.close()
    return plan, refs, results, d


@pytest.mark.parametrize("pairs", [0, 2], ids=["auto", "pairs"])
@pytest.mark.parametrize("shape", [
    # (N, H, W, cin, mid, cout, stride, blocks): few tiles per step (every step in flight at
    # once), and more tiles per step than there are SMs (row blocks completed wave by wave)
    (2, 14, 14, 64, 64, 256, 2, 2),
    (8, 56, 56, 64, 64, 256, 1, 2),
    (4, 28, 28, 256, 128, 512, 2, 2),
], ids=["small", "56x56_b8", "28x28_s2_b4"])
def test_bottleneck_chain_matches_the_oracle_chain(shape, pairs):
    plan, refs, results, d = run_bf16_chain(*shape, seed=9300 + shape[1], graph=False, pairs=pairs)
    assert "out=bf16" in d and "src=1" in d and "res=0" in d, d
    assert f"cta_pairs={1 if pairs == 2 else 0}" in d, d   # narrow or dependent steps: single CTAs unless asked
    for run, outs in enumerate(results):
        for (spec, _, src, rsrc), got, ref in zip(plan, outs, refs):
            assert np.all(np.isfinite(got)), (spec.name, run, "a tile read its input before it was stored")
            ok, worst, frac = chain_close(got, ref)
            assert ok, (spec.name, run, worst, frac)
        assert all(np.array_equal(a, b) for a, b in zip(results[0], outs)), "runs differ"


def test_bottleneck_chain_in_a_graph_repeats_bitwise():
    plan, refs, results, d = run_bf16_chain(2, 28, 28, 64, 64, 256, 2, 2, seed=9400, graph=True)
    for outs in results:
        assert all(np.array_equal(a, b) for a, b in zip(results[0], outs))
        for (spec, *_), got, ref in zip(plan, outs, refs):
            ok, worst, frac = chain_close(got, ref)
            assert ok, (spec.name, worst, frac)


# ------------------------------------------------------------------ refusals

def _pair(out_bf16=True, residual=False):
    spec = S("r", 2, 64, 8, 8, 64, 1, 1)
    inp = inputs_for(spec, 9500)
    return make(spec, inp, out_bf16=out_bf16, residual=residual), to_device_nhwc(inp["x"])


def _refused(steps, status, words):
    with pytest.raises(cf.ConvFusedError) as e:
        cf.ConvChain(steps)
    assert e.value.status == status, str(e.value)
    assert words in str(e.value), str(e.value)


def test_chain_refusals_name_the_reason():
    a, x = _pair()
    b, _ = _pair()
    ya, yb = a.new_output(), b.new_output()
    # a later step writes what an earlier one reads (one launch cannot order that)
    _refused([(a, yb, ya), (b, x, yb)], cf.CONVF_ERR_UNSUPPORTED, "does not come before it")
    # two steps write one buffer
    _refused([(a, x, ya), (b, x, ya)], cf.CONVF_ERR_UNSUPPORTED, "overlapping outputs")
    # a step's input overlaps an earlier output without being that tensor
    big = torch.empty(ya.numel() + 64, dtype=torch.bfloat16, device="cuda")
    _refused([(a, x, big[:ya.numel()].view(ya.shape)), (b, big[8:8 + ya.numel()].view(ya.shape), yb)],
             cf.CONVF_ERR_UNSUPPORTED, "without being exactly")
    # its own output as its input
    _refused([(a, ya, ya)], cf.CONVF_ERR_UNSUPPORTED, "own input")
    # an fp32 output read as the next step's bf16 input
    f, _ = _pair(out_bf16=False)
    yf = f.new_output()
    _refused([(f, x, yf), (b, yf, yb)], cf.CONVF_ERR_UNSUPPORTED, "")
    # mixed output types
    _refused([(a, x, ya), (f, x, yf)], cf.CONVF_ERR_UNSUPPORTED, "output type")
    # a residual handle without its residual, and the reverse
    rh, _ = _pair(residual=True)
    _refused([(rh, x, rh.new_output())], cf.CONVF_ERR_INVALID_ARG, "residual")
    _refused([(a, x, ya, yb)], cf.CONVF_ERR_INVALID_ARG, "residual")
    # a kernel the chain does not run
    spec = S("h", 2, 64, 8, 8, 64, 3, 3, pads=(1, 1, 1, 1))
    inp = inputs_for(spec, 9501)
    halo = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, 3, 3, inp["w"], None, stride=(1, 1),
                        pads=(1, 1, 1, 1), act=ACT_RELU, variant=cf.CONVF_VARIANT_IMPLICIT_GEMM_HALO, out_bf16=True)
    _refused([(halo, x, halo.new_output())], cf.CONVF_ERR_UNSUPPORTED, "variant")
    # a shape mismatch between a producer's output and the consumer's input
    wide, _ = _pair()
    spec2 = S("w", 2, 64, 4, 16, 64, 1, 1)
    inp2 = inputs_for(spec2, 9502)
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp2["bn"]], 1e-5)
    c2 = cf.FusedConv(2, 64, 4, 16, 64, 1, 1, inp2["w"], None, scale, shift, act=ACT_RELU,
                      variant=cf.CONVF_VARIANT_GEMM_1X1, out_bf16=True)
    _refused([(a, x, ya), (c2, ya, c2.new_output())], cf.CONVF_ERR_INVALID_ARG, "is not step 0's output")
    for c in (a, b, f, rh, halo, wide, c2):
        c.close()


def test_chain_allocation_failure_is_reported_and_leaves_nothing_behind():
    a, x = _pair()
    ya = a.new_output()
    for n in (1, 2):   # the chain object, then its device block
        cf.conv_fused_debug_fail_alloc(n)
        _refused([(a, x, ya)], cf.CONVF_ERR_OOM, "(injected)")
    chain = cf.ConvChain([(a, x, ya)])
    chain()
    torch.cuda.synchronize()
    assert chain.status() == cf.CONVF_OK
    chain.close()
    a.close()


# ------------------------------------------------------------------ exact integer chain

@pytest.mark.parametrize("pairs", [1, 2], ids=["single", "pairs"])
def test_integer_chain_is_bit_exact(pairs):
    """Three bottleneck blocks (projection, stride 2, identity shortcuts) on integers: the
    kernel's chain and the oracle's are the same numbers (module docstring)."""
    N, H, W, cin, mid, cout = 4, 30, 30, 64, 64, 128
    plan = bottleneck_chain(N, H, W, cin, mid, cout, 2, 3, seed=9600)
    g = torch.Generator().manual_seed(9599)
    x0 = torch.randint(-16, 17, (N, cin, H, W), generator=g).to(torch.bfloat16)
    x0d = to_device_nhwc(x0)
    convs, ys, steps, ws = [], [], [], []
    for spec, _, src, rsrc in plan:
        fan = spec.C * spec.R * spec.S
        keep = torch.rand((spec.K, spec.C, spec.R, spec.S), generator=g) < 8.0 / fan
        sign = torch.randint(0, 2, keep.shape, generator=g) * 2 - 1
        w = (keep * sign).to(torch.bfloat16)
        conv = cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, w, None, stride=spec.stride,
                            pads=spec.pads, act=cf.CONVF_ACT_CLIP, clip=(-64.0, 64.0), variant=variant_for(spec),
                            out_bf16=True, residual=rsrc is not None)
        y = conv.new_output()
        x = x0d if src < 0 else ys[src]
        steps.append((conv, x, y) if rsrc is None else (conv, x, y, x0d if rsrc < 0 else ys[rsrc]))
        convs.append(conv)
        ys.append(y)
        ws.append(w)
    chain = cf.ConvChain(steps, cta_pairs=pairs)
    refs = []
    for (spec, _, src, rsrc), w in zip(plan, ws):
        x = x0.double().numpy() if src < 0 else refs[src]
        r = None if rsrc is None else (x0.double().numpy() if rsrc < 0 else refs[rsrc])
        refs.append(oracle.conv_bn_act(x, w.double().numpy(), None, None, oracle.ACT_CLIP, -64.0, 64.0,
                                       spec.stride, spec.pads, residual=r))
    assert all(np.all(r == np.round(r)) and np.abs(r).max() <= 64 for r in refs)
    assert any(np.mean(np.abs(r) == 64) < 0.5 for r in refs)   # not everything saturated
    for run in range(2):
        for y in ys:
            y.fill_(float("nan"))
        chain()
        torch.cuda.synchronize()
        assert chain.status() == cf.CONVF_OK
        for (spec, *_), y, ref in zip(plan, ys, refs):
            got = y.cpu().float().contiguous().numpy()
            bad = int(np.sum(got != ref))
            assert bad == 0, (spec.name, run, bad)
    chain.close()
    for c in convs:
        c.close()


# ------------------------------------------------------------------ full-size ResNet-50, batch 32

def _chain_conv(spec, inp, out_bf16=False, residual=False):
    scale, shift = cf.conv_bn_scale_shift(*[t.numpy() for t in inp["bn"]], 1e-5)
    return cf.FusedConv(spec.N, spec.C, spec.H, spec.W, spec.K, spec.R, spec.S, inp["w"], inp["bias"], scale, shift,
                        stride=spec.stride, pads=spec.pads, act=spec.act, variant=variant_for(spec),
                        out_bf16=out_bf16, residual=residual)


def test_resnet50_b32_chain_every_output():
    """The benchmark's chain: the 52 non-stem ResNet-50 layers at batch 32, each on its own seeded
    input (the benchmark's seeds), fp32 outputs, one launch; every output of every layer against
    the oracle within the single-conv bound."""
    specs = workloads.resnet50_layers(32)
    steps, ins = [], []
    for i, spec in enumerate(specs[1:], 1):
        inp = inputs_for(spec, synthetic.seed_for(3, i))
        conv = _chain_conv(spec, inp)
        steps.append((conv, to_device_nhwc(inp["x"]), conv.new_output()))
        ins.append(inp)
    chain = cf.ConvChain(steps)
    for _, _, y in steps:
        y.fill_(float("nan"))
    chain()
    torch.cuda.synchronize()
    assert chain.status() == cf.CONVF_OK
    worst_all = 0.0
    for (conv, _, y), spec, inp in zip(steps, specs[1:], ins):
        ok, worst, idx = compare(y.cpu().contiguous().numpy(), oracle_step(spec, inp["x"].double().numpy(), inp),
                                 False)
        assert ok, (spec.name, worst, idx)
        worst_all = max(worst_all, worst)
    print(f"52-step chain, every output: worst |d|/allowance = {worst_all:.4g}")
    chain.close()
    for conv, _, _ in steps:
        conv.close()


def test_resnet50_b32_network_chain():
    """ResNet-50's own dataflow at batch 32 as one dependent chain (bf16 activations, residuals,
    the residual branch's BN damped as in synthetic.residual_branch_inputs): every output of every
    layer against the oracle's chain (bf16-rounded intermediates) within the bottleneck-chain
    bound."""
    specs = workloads.resnet50_layers(32)
    flow = workloads.resnet50_dataflow()
    g = torch.Generator().manual_seed(7001)
    x0 = torch.randn((32, 64, 56, 56), generator=g).to(torch.bfloat16)
    x0d = to_device_nhwc(x0)
    steps, ys, ins = [], [], []
    for li, src, rsrc in flow:
        # a block's last conv (the one adding the shortcut) with the damped residual-branch BN
        gen = synthetic.residual_branch_inputs if rsrc is not None else synthetic.conv_inputs
        inp = gen(specs[li], synthetic.seed_for(3, li))
        conv = _chain_conv(specs[li], inp, out_bf16=True, residual=rsrc is not None)
        y = conv.new_output()
        x = x0d if src < 0 else ys[src]
        steps.append((conv, x, y) if rsrc is None else (conv, x, y, x0d if rsrc < 0 else ys[rsrc]))
        ys.append(y)
        ins.append(inp)
    chain = cf.ConvChain(steps)
    for y in ys:
        y.fill_(float("nan"))
    chain()
    torch.cuda.synchronize()
    assert chain.status() == cf.CONVF_OK
    refs = []
    worst_all, frac_all = 0.0, 0.0
    for k, ((li, src, rsrc), y, inp) in enumerate(zip(flow, ys, ins)):
        x = x0.double().numpy() if src < 0 else refs[src].astype(np.float64)
        r = None if rsrc is None else (x0.double().numpy() if rsrc < 0 else refs[rsrc].astype(np.float64))
        ref = oracle.round_bf16(oracle_step(specs[li], x, inp, residual=r))
        refs.append(ref.astype(np.float32))   # bf16 values are exact in float32
        got = y.cpu().float().contiguous().numpy()
        assert np.all(np.isfinite(got)), (specs[li].name, "a tile read its input before it was stored")
        ok, worst, frac = chain_close(got, ref)
        assert ok, (specs[li].name, worst, frac)
        worst_all, frac_all = max(worst_all, worst), max(frac_all, frac)
    print(f"ResNet-50 network chain: worst ratio {worst_all:.3g}, largest share > 1 unit {frac_all:.3g}")
    chain.close()
    for st in steps:
        st[0].close()
