"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds none of the method's arithmetic: it draws random bytes and
random normals and names the workloads.  An IQ4_XS weight matrix is produced
as raw super-block bytes -- the fp16 ``d`` field is drawn as |N(0,1)| * scale
and stored at bytes 0-1 of each 136-byte block; every other byte (scales_h,
scales_l, qs) is uniform, which makes each 6-bit ``ls`` uniform on 0..63 and
each nibble uniform on 0..15 whatever the bit order inside the block.

Stream order for one matrix: the block ``d`` normals (row-major block order),
then the other 134 bytes of every block, then the activations.
"""
from __future__ import annotations

import dataclasses

import numpy as np

QK = 256
BLOCK_BYTES = 136


def iq4xs_weights(rng: np.random.Generator, N: int, K: int, d_scale: float) -> np.ndarray:
    """Random IQ4_XS matrix [N][K/256] super-blocks as uint8 [N, K/256*136]."""
    if K % QK:
        raise ValueError("K must be a multiple of 256")
    nb = N * (K // QK)
    d = (np.abs(rng.standard_normal(nb)) * d_scale).astype(np.float16)
    rest = rng.integers(0, 256, size=(nb, BLOCK_BYTES - 2), dtype=np.uint8)
    blocks = np.empty((nb, BLOCK_BYTES), dtype=np.uint8)
    blocks[:, 0:2] = d.view(np.uint8).reshape(nb, 2)  # little-endian fp16 bits
    blocks[:, 2:] = rest
    return blocks.reshape(N, (K // QK) * BLOCK_BYTES)


SUB = 32
B18_BYTES = 18


def block32_weights(rng: np.random.Generator, N: int, K: int, d_scale: float) -> np.ndarray:
    """Random matrix of 18-byte, 32-weight blocks (the Q4_0 and IQ4_NL byte
    shape: fp16 ``d`` at bytes 0-1 drawn as |N(0,1)| * scale, then 16 uniform
    bytes of nibbles) as uint8 [N, K/32*18].  Stream order: the ``d`` normals,
    then the nibble bytes, both in row-major block order."""
    if K % SUB:
        raise ValueError("K must be a multiple of 32")
    nb = N * (K // SUB)
    d = (np.abs(rng.standard_normal(nb)) * d_scale).astype(np.float16)
    qs = rng.integers(0, 256, size=(nb, B18_BYTES - 2), dtype=np.uint8)
    blocks = np.empty((nb, B18_BYTES), dtype=np.uint8)
    blocks[:, 0:2] = d.view(np.uint8).reshape(nb, 2)
    blocks[:, 2:] = qs
    return blocks.reshape(N, (K // SUB) * B18_BYTES)


# Weight formats by name: IQ4_XS (256-weight super-blocks of 136 bytes), Q4_0
# and IQ4_NL (32-weight blocks of 18 bytes; the same bytes decode either way).
WTYPES = {"iq4_xs": 0, "q4_0": 1, "iq4_nl": 2}


def weights_for(wtype: int, rng: np.random.Generator, N: int, K: int,
                d_scale: float) -> np.ndarray:
    """Random weights in the byte shape of format ``wtype``."""
    if wtype == 0:
        return iq4xs_weights(rng, N, K, d_scale)
    return block32_weights(rng, N, K, d_scale)


def activations(rng: np.random.Generator, M: int, K: int, outlier_frac: float = 0.0,
                outlier_scale: float = 20.0, bf16_round: bool = False) -> np.ndarray:
    """x fp32 [M, K] ~ N(0,1).  ``outlier_frac`` of the channels (chosen without
    replacement, the same for every row) are multiplied by ``outlier_scale``;
    ``bf16_round`` rounds every value to bfloat16 (RNE) and widens it back."""
    x = rng.standard_normal((M, K), dtype=np.float32)
    n_out = int(np.floor(outlier_frac * K))
    if n_out:
        ch = rng.choice(K, size=n_out, replace=False)
        x[:, ch] *= np.float32(outlier_scale)
    if bf16_round:
        import torch
        x = torch.from_numpy(x).to(torch.bfloat16).to(torch.float32).numpy()
    return np.ascontiguousarray(x)


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic workload: weight shapes, batch sizes and input recipe."""
    name: str
    seed: int
    shapes: tuple          # ((N, K), ...)
    ms: tuple              # batch sizes M
    d_scale: float
    outlier_frac: float = 0.0
    bf16_round: bool = False
    layers: int = 1        # >1: the shapes repeat per decoder layer

    def rng(self, shape_index: int = 0, layer: int = 0) -> np.random.Generator:
        return np.random.default_rng([self.seed, shape_index, layer])

    def weights(self, shape_index: int = 0, layer: int = 0) -> np.ndarray:
        N, K = self.shapes[shape_index]
        return iq4xs_weights(self.rng(shape_index, layer), N, K, self.d_scale)

    def inputs(self, shape_index: int = 0, M: int | None = None, layer: int = 0):
        """(W bytes, x [M,K]) drawn from one stream: W first, then x.  Smaller
        M are prefixes of the largest one when drawn with M=max(ms)."""
        N, K = self.shapes[shape_index]
        rng = self.rng(shape_index, layer)
        w = iq4xs_weights(rng, N, K, self.d_scale)
        M = max(self.ms) if M is None else M
        x = activations(rng, M, K, self.outlier_frac, bf16_round=self.bf16_round)
        return w, x


# Workloads of the method's decode/verify batch range, named by what they are.
TINY = Workload("tiny_256x1024", seed=0, shapes=((256, 1024),), ms=(1, 4, 8), d_scale=2e-3)
SQUARE = Workload("square_4096x4096", seed=1, shapes=((4096, 4096),),
                  ms=(1, 2, 4, 8, 12, 16, 32, 64, 96), d_scale=1e-3)
DECODER_27B = Workload(
    "decoder27b_9proj", seed=2,
    shapes=((5120, 5120), (6144, 5120), (1024, 5120), (10240, 5120), (12288, 5120),
            (5120, 6144), (17408, 5120), (34816, 5120), (5120, 17408)),
    ms=(1, 4, 8, 16, 64), d_scale=2e-3, outlier_frac=0.01)
PREFILL = Workload("prefill_sweep", seed=3, shapes=((17408, 5120), (5120, 17408)),
                   ms=(96, 128, 192, 256, 512), d_scale=2e-3, bf16_round=True)
DECODE_STREAM = Workload(
    "decode_stream_64layers", seed=4,
    shapes=((12288, 5120), (5120, 6144), (34816, 5120), (5120, 17408)),
    ms=(1, 2, 8, 16, 32), d_scale=2e-3, layers=64)

WORKLOADS = {w.name: w for w in (TINY, SQUARE, DECODER_27B, PREFILL, DECODE_STREAM)}


@dataclasses.dataclass(frozen=True)
class MoEWorkload:
    """Routed experts of one layer: G experts of shape (N, K); each of T
    tokens is routed to ``topk`` distinct experts drawn uniformly; the
    activation rows are grouped by expert (expert g owns rows
    [row_offsets[g], row_offsets[g+1]), tokens in increasing order)."""
    name: str
    seed: int
    G: int
    N: int
    K: int
    topk: int
    tokens: tuple
    d_scale: float

    def weights(self) -> np.ndarray:
        """uint8 [G, N, K/256*136]; expert g from its own stream."""
        return np.stack([iq4xs_weights(np.random.default_rng([self.seed, g]), self.N, self.K,
                                       self.d_scale) for g in range(self.G)])

    def routing(self, T: int):
        """(row_offsets int32 [G+1], token of each row int64 [T*topk])."""
        rng = np.random.default_rng([self.seed, 100000 + T])
        choice = np.stack([rng.choice(self.G, size=self.topk, replace=False) for _ in range(T)])
        tok = np.repeat(np.arange(T), self.topk)
        exp = choice.reshape(-1)
        order = np.lexsort((tok, exp))  # by expert, then token
        counts = np.bincount(exp, minlength=self.G)
        offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
        return offsets, tok[order]

    def inputs(self, T: int):
        """(x [T, K] token activations, rows [T*topk, K] grouped by expert,
        row_offsets int32 [G+1])."""
        rng = np.random.default_rng([self.seed, 200000 + T])
        x = activations(rng, T, self.K)
        offsets, tok = self.routing(T)
        return x, np.ascontiguousarray(x[tok]), offsets


# A routed-expert layer for the grouped matmul (decode: a few tokens, top-8 of
# 128 experts; 214 MB of expert weights, larger than L2).
MOE_DECODE = MoEWorkload("moe_decode_128x1536x2048", seed=5, G=128, N=1536, K=2048, topk=8,
                         tokens=(1, 4, 16), d_scale=2e-3)
