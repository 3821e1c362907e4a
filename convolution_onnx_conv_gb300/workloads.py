"""Layer shape tables for the synthetic workloads (shapes only, no arithmetic).

The pages benchmark whole ONNX models (ResNet50-v2 in "tensorforge", section
"Engine latency"; MobileNetV2 in "onnx-vulkan-rs") whose model files are not
available here, so the workloads are the conv layers of the public
architectures, with seeded synthetic tensors of those shapes.
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace
from typing import List, Optional, Tuple

ACT_NONE, ACT_RELU, ACT_RELU6, ACT_CLIP = 0, 1, 2, 3


@dataclass(frozen=True)
class ConvSpec:
    """One ONNX Conv node: x[N][C][H][W], W[K][C/group][R][S]."""
    name: str
    N: int
    C: int
    H: int
    W: int
    K: int
    R: int
    S: int
    stride: Tuple[int, int] = (1, 1)
    pads: Tuple[int, int, int, int] = (0, 0, 0, 0)   # h_begin, w_begin, h_end, w_end
    dilation: Tuple[int, int] = (1, 1)
    group: int = 1
    act: int = ACT_RELU
    has_bias: bool = False
    has_bn: bool = True
    dtype: str = "bf16"            # "bf16" or "s8"
    values: str = "normal"         # "uniform" (U[-1,1]) or "normal" (N(0,1), He weights)

    @property
    def out_hw(self) -> Tuple[int, int]:
        sh, sw = self.stride
        dh, dw = self.dilation
        pt, pl, pb, pr = self.pads
        ho = (self.H + pt + pb - dh * (self.R - 1) - 1) // sh + 1
        wo = (self.W + pl + pr - dw * (self.S - 1) - 1) // sw + 1
        return ho, wo

    @property
    def flops(self) -> int:
        """2*N*K*Ho*Wo*(C/group)*R*S: every tap counted, padded ones included."""
        ho, wo = self.out_hw
        return 2 * self.N * self.K * ho * wo * (self.C // self.group) * self.R * self.S

    @property
    def algorithmic_bytes(self) -> int:
        """x once + W once + per-channel epilogue vectors + y once."""
        ho, wo = self.out_hw
        if self.dtype == "s8":
            xb, wb, yb, vec = 1, 1, 1, 12          # int32 bias, multiplier, shift
        else:
            xb, wb, yb, vec = 2, 2, 4, 8           # fp32 scale + bias
            if self.group == self.C and self.group == self.K:
                wb = 4                             # depthwise taps are folded fp32
        return (self.N * self.C * self.H * self.W * xb
                + self.K * (self.C // self.group) * self.R * self.S * wb
                + self.K * vec + self.N * self.K * ho * wo * yb)

    def with_batch(self, n: int) -> "ConvSpec":
        return replace(self, N=n, name=f"{self.name.split('@')[0]}@b{n}")


def _pad(r: int) -> Tuple[int, int, int, int]:
    p = r // 2
    return (p, p, p, p)


def single_conv_relu() -> ConvSpec:
    """N=1, C=16, 32x32, K=32 3x3 s1 p1: bias + ReLU, no BN, uniform values."""
    return ConvSpec("conv3x3_c16k32_32x32", 1, 16, 32, 32, 32, 3, 3, (1, 1), (1, 1, 1, 1),
                    act=ACT_RELU, has_bias=True, has_bn=False, values="uniform")


def bottleneck_1x1(n: int = 32) -> List[ConvSpec]:
    """ResNet-50 bottleneck 1x1 reduce / expand at 56x56: 256->64 and 64->256."""
    return [ConvSpec(f"r50_1x1_256to64_56@b{n}", n, 256, 56, 56, 64, 1, 1),
            ConvSpec(f"r50_1x1_64to256_56@b{n}", n, 64, 56, 56, 256, 1, 1)]


def resnet50_layers(n: int = 32) -> List[ConvSpec]:
    """The 53 conv layers of ResNet-50 (v2 / gluon convention: stride on the 3x3
    conv and on the 1x1 projection), 224x224 input, stem 7x7/2 pad 3."""
    L: List[ConvSpec] = []

    def add(tag, c, h, k, r, s):
        L.append(ConvSpec(f"r50_{len(L):02d}_{tag}@b{n}", n, c, h, h, k, r, r, (s, s), _pad(r)))

    add("stem7x7", 3, 224, 64, 7, 2)
    cin, h = 64, 56
    for stage, (mid, blocks) in enumerate(((64, 3), (128, 4), (256, 6), (512, 3))):
        out = mid * 4
        for b in range(blocks):
            s = 2 if (b == 0 and stage > 0) else 1
            add(f"s{stage}b{b}_1x1a", cin, h, mid, 1, 1)
            add(f"s{stage}b{b}_3x3", mid, h, mid, 3, s)
            ho = h // s
            add(f"s{stage}b{b}_1x1b", mid, ho, out, 1, 1)
            if b == 0:
                add(f"s{stage}b{b}_proj", cin, h, out, 1, s)
            cin, h = out, ho
    assert len(L) == 53
    return L


def resnet50_dataflow() -> List[Tuple[int, int, Optional[int]]]:
    """The bottleneck layers of ``resnet50_layers`` (all but the stem) in an order in which every
    layer comes after the layers it reads, as ``(layer, src, rsrc)``: the index into
    ``resnet50_layers`` and the positions in this list of the layers whose outputs are its input
    (``src``) and the residual added in its epilogue (``rsrc``: each block's last 1x1 conv adds
    the block's shortcut, the projection's output or the block input), -1 standing for the
    stack's input (the stem's 56x56x64 output after max pooling) and ``rsrc`` None for no
    residual.  Per block: the projection (first block of a stage), the 1x1 reduce, the 3x3, the
    1x1 expand."""
    names = [s.name.split("_", 2)[2].split("@")[0] for s in resnet50_layers(1)]
    index = {n: i for i, n in enumerate(names)}
    out: List[Tuple[int, int, Optional[int]]] = []
    block_in = -1
    for stage, (mid, blocks) in enumerate(((64, 3), (128, 4), (256, 6), (512, 3))):
        for b in range(blocks):
            pre = f"s{stage}b{b}"
            shortcut = block_in
            if pre + "_proj" in index:
                out.append((index[pre + "_proj"], block_in, None))
                shortcut = len(out) - 1
            out.append((index[pre + "_1x1a"], block_in, None))
            out.append((index[pre + "_3x3"], len(out) - 1, None))
            out.append((index[pre + "_1x1b"], len(out) - 1, shortcut))
            block_in = len(out) - 1
    return out


MOBILENETV2_BLOCKS = [  # (C_in, hidden, C_out, H_in, stride)
    (32, 32, 16, 112, 1),
    (16, 96, 24, 112, 2),
    (24, 144, 24, 56, 1),
    (24, 144, 32, 56, 2),
    (32, 192, 32, 28, 1), (32, 192, 32, 28, 1),
    (32, 192, 64, 28, 2),
    (64, 384, 64, 14, 1), (64, 384, 64, 14, 1), (64, 384, 64, 14, 1),
    (64, 384, 96, 14, 1),
    (96, 576, 96, 14, 1), (96, 576, 96, 14, 1),
    (96, 576, 160, 14, 2),
    (160, 960, 160, 7, 1), (160, 960, 160, 7, 1),
    (160, 960, 320, 7, 1),
]


def mobilenetv2_layers(n: int = 64) -> List[ConvSpec]:
    """The 17 inverted-residual blocks of MobileNetV2 (width 1.0, 224x224 input):
    1x1 expand + ReLU6 (absent in block 0, t=1), depthwise 3x3 pad 1 + ReLU6,
    1x1 project with no activation (linear bottleneck)."""
    L: List[ConvSpec] = []
    for i, (cin, hid, cout, h, s) in enumerate(MOBILENETV2_BLOCKS):
        if hid != cin:
            L.append(ConvSpec(f"mv2_{i:02d}_expand@b{n}", n, cin, h, h, hid, 1, 1,
                              act=ACT_RELU6))
        L.append(ConvSpec(f"mv2_{i:02d}_dw_s{s}@b{n}", n, hid, h, h, hid, 3, 3, (s, s),
                          (1, 1, 1, 1), group=hid, act=ACT_RELU6))
        ho = (h + 2 - 3) // s + 1
        L.append(ConvSpec(f"mv2_{i:02d}_project@b{n}", n, hid, ho, ho, cout, 1, 1,
                          act=ACT_NONE))
    return L


def mobilenetv2_blocks(n: int = 64):
    """The 17 blocks as (name, N, Cin, H, Ch, Cout, stride, expand, residual): the skip connection
    where the block keeps its stride at 1 and its channel count (the public architecture)."""
    return [(f"mv2_block{i:02d}@b{n}", n, cin, h, hid, cout, s, hid != cin, s == 1 and cin == cout)
            for i, (cin, hid, cout, h, s) in enumerate(MOBILENETV2_BLOCKS)]


def depthwise_layers(n: int = 64) -> List[ConvSpec]:
    return [l for l in mobilenetv2_layers(n) if l.group > 1]


RESNEXT_GROUPED = [  # (width, H_in, stride): the grouped 3x3 of each ResNeXt-50 32x4d stage
    (128, 56, 1), (256, 56, 2), (512, 28, 2), (1024, 14, 2),
]


def resnext50_grouped_layers(n: int = 32) -> List[ConvSpec]:
    """The grouped 3x3 convs of ResNeXt-50 (32x4d): 32 groups of 4, 8, 16 and 32 channels, the
    first block of stages 2-4 strided on the 3x3, folded BN + ReLU."""
    return [ConvSpec(f"rx50_3x3_g32_c{c}_{h}_s{s}@b{n}", n, c, h, h, c, 3, 3, (s, s), (1, 1, 1, 1), group=32)
            for c, h, s in RESNEXT_GROUPED]


INT8_SHAPES = [  # (C = K, H_in, stride): the seven distinct ResNet-50 3x3 shapes
    (64, 56, 1), (128, 56, 2), (128, 28, 1), (256, 28, 2), (256, 14, 1), (512, 14, 2),
    (512, 7, 1),
]


def int8_layers(n: int = 64) -> List[ConvSpec]:
    return [ConvSpec(f"s8_3x3_c{c}_{h}_s{s}@b{n}", n, c, h, h, c, 3, 3, (s, s), (1, 1, 1, 1),
                     act=ACT_RELU, has_bias=True, has_bn=False, dtype="s8", values="int")
            for c, h, s in INT8_SHAPES]
