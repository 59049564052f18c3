"""Layer-shaped gradient layouts used by the workloads.

transformer_shapes: the Transformer of "How GPipe works" (GPipe page, section 1,
the parameter-count formula P(L) ~ 2Vd + L(4d^2 + 2dh + biases, LN) with
d=2048, h=8192, V=32000).  Reading of the unlisted parts: per layer
LN1 (gain, bias), Q/K/V/O weights d x d with d-sized biases, LN2 (gain, bias),
FFN weights d x h and h x d with biases; an input embedding and an output
softmax projection, each V x d.  Forward order.

resnet18_shapes: ResNet-18's conv/BN/fc tensors ("[AI System] Training With
Multiple GPUs", section Memory: ResNet-18 has about 11.7M parameters).
Reading: the standard ResNet-18 (7x7 stem, four stages of two basic blocks
with 64/128/256/512 channels, 1x1 downsample in stages 2-4, a BN gain and
bias per conv, a 1000-way fc with bias).  Forward order.
"""
from __future__ import annotations

from math import prod


def transformer_shapes(layers: int = 24, d: int = 2048, h: int = 8192, vocab: int = 32000):
    out = [("embed", (vocab, d))]
    for l in range(layers):
        p = "layer%d." % l
        out += [
            (p + "ln1.gain", (d,)), (p + "ln1.bias", (d,)),
            (p + "attn.q.weight", (d, d)), (p + "attn.q.bias", (d,)),
            (p + "attn.k.weight", (d, d)), (p + "attn.k.bias", (d,)),
            (p + "attn.v.weight", (d, d)), (p + "attn.v.bias", (d,)),
            (p + "attn.o.weight", (d, d)), (p + "attn.o.bias", (d,)),
            (p + "ln2.gain", (d,)), (p + "ln2.bias", (d,)),
            (p + "ffn.w1", (d, h)), (p + "ffn.b1", (h,)),
            (p + "ffn.w2", (h, d)), (p + "ffn.b2", (d,)),
        ]
    out.append(("softmax", (vocab, d)))
    return out


def resnet18_shapes(num_classes: int = 1000):
    out = [("conv1.weight", (64, 3, 7, 7)), ("bn1.weight", (64,)), ("bn1.bias", (64,))]
    cin = 64
    for stage, cout in enumerate((64, 128, 256, 512), start=1):
        for blk in range(2):
            p = "layer%d.%d." % (stage, blk)
            first_in = cin if blk == 0 else cout
            out += [
                (p + "conv1.weight", (cout, first_in, 3, 3)), (p + "bn1.weight", (cout,)), (p + "bn1.bias", (cout,)),
                (p + "conv2.weight", (cout, cout, 3, 3)), (p + "bn2.weight", (cout,)), (p + "bn2.bias", (cout,)),
            ]
            if blk == 0 and first_in != cout:
                out += [(p + "downsample.0.weight", (cout, first_in, 1, 1)),
                        (p + "downsample.1.weight", (cout,)), (p + "downsample.1.bias", (cout,))]
        cin = cout
    out += [("fc.weight", (num_classes, 512)), ("fc.bias", (num_classes,))]
    return out


def numels(shapes):
    return [prod(s) for _, s in shapes]
