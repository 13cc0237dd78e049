"""Seeded synthetic inputs for the quantized-linear workloads.

This module only draws random numbers and lays them out; it contains none of
the layer's arithmetic (no scales, no quantization, no matmul).  Both the CUDA
path and the CPU oracle consume what it produces.

Recipe (shapes and distributions follow the workloads the serving pages
measure: Qwen2.5-3B / 7B-class linear shapes, decode M <= 256, prefill M >= 1024):
  * weights: fp32 ~ N(0, 1/K), row-major [N, K] (nn.Linear layout);
  * activations: BF16 (round-to-nearest-even of fp32 draws) ~ N(0, 1), row-major
    [M, K]; where a workload asks for outliers, round(K/100) channels chosen by a
    seeded permutation of K (a property of the layer, shared by the calibration
    and run-time batches) are multiplied by 20 before the BF16 rounding;
  * calibration batch: 64 x 512 = 32768 rows from the same distribution, drawn
    from its own seed;
  * bias: BF16 ~ N(0, 0.01) read as variance 0.01 (std 0.1);
  * seeds: base seed 0, one sub-seed per (workload, layer, tensor, role).
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

BASE_SEED = 0
CALIB_ROWS = 64 * 512


def sub_seed(workload: str, layer: int, tensor: str, role: str) -> int:
    h = hashlib.blake2b(f"{workload}/{layer}/{tensor}/{role}".encode(), digest_size=8)
    return int.from_bytes(h.digest(), "little")


def rng_for(workload: str, layer: int, tensor: str, role: str) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence(
        [BASE_SEED, sub_seed(workload, layer, tensor, role)])))


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to BF16 (nearest, ties to even) and return the 16-bit patterns."""
    u = np.ascontiguousarray(a, np.float32).view(np.uint32)
    r = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return r.astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.ascontiguousarray(b, np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def outlier_channels(K: int, rng: np.random.Generator) -> np.ndarray:
    n_out = int(round(K / 100.0))
    return np.sort(rng.permutation(K)[:n_out])


def weights(N: int, K: int, rng: np.random.Generator) -> np.ndarray:
    w = rng.standard_normal((N, K), dtype=np.float32)
    w *= np.float32(1.0 / np.sqrt(K))
    return w


def activations(M: int, K: int, rng: np.random.Generator, outliers: np.ndarray | None = None,
                scale: float = 20.0, chunk_rows: int = 4096) -> np.ndarray:
    """BF16 bits [M, K]; generated in row chunks to bound host memory."""
    out = np.empty((M, K), np.uint16)
    for r0 in range(0, M, chunk_rows):
        r1 = min(M, r0 + chunk_rows)
        a = rng.standard_normal((r1 - r0, K), dtype=np.float32)
        if outliers is not None and outliers.size:
            a[:, outliers] *= np.float32(scale)
        out[r0:r1] = f32_to_bf16_bits(a)
    return out


def bias(N: int, rng: np.random.Generator, std: float = 0.1) -> np.ndarray:
    return f32_to_bf16_bits(rng.standard_normal(N, dtype=np.float32) * np.float32(std))


# --------------------------------------------------------------------------
# Workloads (shapes and distributions as described above)
# --------------------------------------------------------------------------
@dataclass
class Linear:
    name: str          # e.g. "q_proj"
    K: int
    N: int
    M: int
    qtype: str         # "int8" | "e4m3"
    form: str          # "w8a16" | "w8a8"
    bias: bool = False
    outliers: bool = False
    workload: str = ""
    layer: int = 0
    glu: bool = False  # merged gate_up [N = 2I, K] with the SiLU * up epilogue: output [M, N/2]


@dataclass
class Workload:
    name: str
    desc: str
    linears: list[Linear] = field(default_factory=list)


SMALL = "int8-w8a16-1k"            # INT8 W8A16, K=N=1024, M in {1,16}
DECODE7B = "e4m3-w8a16-decode-7b"  # FP8-E4M3 W8A16 decode sweep, 7B-class shapes
W8A8_3B = "int8-w8a8-static-3b"    # INT8 W8A8 static, 3B-class shapes, bias
PREFILL = "e4m3-w8a8-static-prefill"  # FP8-E4M3 W8A8 static prefill
W8A8_DYN_3B = "int8-w8a8-dynamic-3b"  # INT8 W8A8 with dynamic per-token scales, 3B-class shapes, bias
STACK = "stack-36L-3b"             # 36-layer 3B linear stack, decode + prefill


def workload(name: str) -> Workload:
    if name == SMALL:
        return Workload(name, "INT8 W8A16 single linear K=N=1024, M in {1,16}, no bias",
                        [Linear("linear", 1024, 1024, M, "int8", "w8a16", workload=name)
                         for M in (1, 16)])
    if name == DECODE7B:
        shapes = [("q_proj", 3584, 3584), ("gate_up_proj", 3584, 37888), ("down_proj", 18944, 3584)]
        return Workload(name, "FP8-E4M3 W8A16 decode sweep, hidden 3584 / intermediate 18944",
                        [Linear(s, K, N, M, "e4m3", "w8a16", outliers=True, workload=name)
                         for M in (1, 8, 32, 128, 256) for (s, K, N) in shapes])
    if name == W8A8_3B:
        shapes = [("q_proj", 1, 2048, 2048), ("up_proj", 16, 2048, 11008),
                  ("down_proj", 256, 11008, 2048), ("up_proj", 1024, 2048, 11008)]
        return Workload(name, "INT8 W8A8 static, 3B-class microbench shapes, bias",
                        [Linear(s, K, N, M, "int8", "w8a8", bias=True, workload=name)
                         for (s, M, K, N) in shapes])
    if name == W8A8_DYN_3B:
        shapes = [("q_proj", 1, 2048, 2048), ("up_proj", 16, 2048, 11008),
                  ("down_proj", 256, 11008, 2048), ("up_proj", 1024, 2048, 11008)]
        return Workload(name, "INT8 W8A8 dynamic per-token, 3B-class microbench shapes, bias",
                        [Linear(s, K, N, M, "int8", "w8a8dyn", bias=True, workload=name)
                         for (s, M, K, N) in shapes])
    if name == PREFILL:
        kn = [(2048, 11008), (11008, 2048), (2048, 2048)]
        return Workload(name, "FP8-E4M3 W8A8 static prefill",
                        [Linear(f"k{K}_n{N}", K, N, M, "e4m3", "w8a8", outliers=True, workload=name)
                         for M in (1024, 4096, 16384, 32640) for (K, N) in kn])
    raise KeyError(name)


STACK_LAYERS = 36
STACK_SHAPES = [("q_proj", 2048, 2048), ("k_proj", 2048, 256), ("v_proj", 2048, 256),
                ("o_proj", 2048, 2048), ("gate_up_proj", 2048, 22016), ("down_proj", 11008, 2048)]


# The same layer with the merged projections of the model's four quantized linears
# per layer (tiny-vLLM README, quality check: 112 target layers for 28 layers):
# merged qkv, o, merged gate_up with the SiLU * up epilogue, down.
STACK_FUSED_SHAPES = [("qkv_proj", 2048, 2560, False), ("o_proj", 2048, 2048, False),
                      ("gate_up_silu", 2048, 22016, True), ("down_proj", 11008, 2048, False)]


def stack_linears(phase: str, fused: bool = False) -> list[Linear]:
    """36 layers x 6 linears (or x 4 merged ones when fused); decode = INT8 W8A16 at
    M=256, prefill = E4M3 W8A8 at M=8192."""
    if phase == "decode":
        M, qt, form = 256, "int8", "w8a16"
    elif phase == "prefill":
        M, qt, form = 8192, "e4m3", "w8a8"
    else:
        raise KeyError(phase)
    if fused:
        return [Linear(s, K, N, M, qt, form, workload=f"{STACK}-fused-{phase}", layer=l, glu=g)
                for l in range(STACK_LAYERS) for (s, K, N, g) in STACK_FUSED_SHAPES]
    return [Linear(s, K, N, M, qt, form, workload=f"{STACK}-{phase}", layer=l)
            for l in range(STACK_LAYERS) for (s, K, N) in STACK_SHAPES]


def make_inputs(lin: Linear, want=("w", "x", "cal", "bias"), x_rows: int | None = None):
    """Draw the tensors of one linear.  Returns a dict with any of:
    w  fp32 [N,K];  x  BF16 bits [M,K] (or x_rows rows);  cal BF16 bits [32768,K]
    (W8A8 only);  bias BF16 bits [N] (when the workload has one)."""
    wl, L = lin.workload, lin.layer
    out = {}
    outl = None
    if lin.outliers:
        outl = outlier_channels(lin.K, rng_for(wl, L, f"{lin.name}.K{lin.K}", "outliers"))
    if "w" in want:
        out["w"] = weights(lin.N, lin.K, rng_for(wl, L, f"{lin.name}.K{lin.K}.N{lin.N}", "weight"))
    if "x" in want:
        M = lin.M if x_rows is None else x_rows
        out["x"] = activations(M, lin.K, rng_for(wl, L, f"{lin.name}.K{lin.K}.M{lin.M}", "act"), outl)
    if "cal" in want and lin.form == "w8a8":  # static W8A8 only; the dynamic form needs no calibration
        out["cal"] = activations(CALIB_ROWS, lin.K, rng_for(wl, L, f"{lin.name}.K{lin.K}", "calib"), outl)
    if "bias" in want and lin.bias:
        out["bias"] = bias(lin.N, rng_for(wl, L, f"{lin.name}.N{lin.N}", "bias"))
    return out


# --------------------------------------------------------------------------
# Mixed KV-cache workload: Qwen2.5-7B attention KV (28 layers, 4 kv heads,
# head_dim 128) in a paged cache of 256-token blocks.  One step per layer:
# an 8192-token prefill chunk is quantized into freshly allocated blocks, and
# the layer's whole 32768-token context is read back as BF16 (the attention
# read).  Block ids come from a seeded permutation (a block allocator hands out
# non-contiguous blocks; tokens are contiguous inside a block).
# --------------------------------------------------------------------------
KV7B = "kv-mixed-7b"
KV_LAYERS, KV_HEADS, KV_HEAD_DIM, KV_BLOCK = 28, 4, 128, 256
KV_CHUNK, KV_CONTEXT = 8192, 32768


def kv_block_table(layer: int, n_blocks: int = KV_CONTEXT // KV_BLOCK) -> np.ndarray:
    return rng_for(KV7B, layer, "block_table", "perm").permutation(n_blocks)


def kv_slots(blocks: np.ndarray, block: int = KV_BLOCK) -> np.ndarray:
    """int64 slots of the tokens of the given blocks, in order."""
    return (np.asarray(blocks, np.int64)[:, None] * block + np.arange(block, dtype=np.int64)[None, :]).reshape(-1)


def kv_chunk_slots(layer: int) -> np.ndarray:
    """Slots of the layer's prefill chunk: the first KV_CHUNK/KV_BLOCK blocks of its table."""
    return kv_slots(kv_block_table(layer)[:KV_CHUNK // KV_BLOCK])


def kv_context_slots(layer: int) -> np.ndarray:
    """Slots of the layer's whole context, in block-table order."""
    return kv_slots(kv_block_table(layer))


def kv_tokens(layer: int, T: int, role: str) -> np.ndarray:
    """BF16 bits [T, H*D] of new key or value rows, N(0,1) with 1% outlier channels x20."""
    rng = rng_for(KV7B, layer, f"{role}.T{T}", "act")
    outl = outlier_channels(KV_HEADS * KV_HEAD_DIM, rng_for(KV7B, layer, role, "outliers"))
    return activations(T, KV_HEADS * KV_HEAD_DIM, rng, outl)
