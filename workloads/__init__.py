"""Seeded synthetic workloads for paged-KV decode attention.

This module only builds inputs.  It holds none of the attention arithmetic and
imports neither the CUDA library nor the oracle; both the tests and the bench
use it so that the GPU path and the CPU oracle read the very same bits.

Five named workloads follow the shapes of a paged KV cache used in decode
(the "Decode-only block-table attention" and "Physical KV blocks with logical
per-request block tables" items of the ForgeLLM README's feature list, and
the "Why paged KV cache?" section of the LLM-Inference-Engine README):

  tiny         4 seqs, 4 q / 2 kv heads, D=64,  bs=16, L={1,17,33,64}, pool 32
  tinyllama    8 seqs, 32 / 4,             D=64,  bs=16, L~U[128,2048], pool 2x
  cont_batch  64 seqs, 32 / 32 (MHA),      D=128, bs=16, L~logU[16,4096],
              one appended token per seq (8 slots = -1), 1% key rows x8
  llama3_8b  256 seqs, 32 / 8,             D=128, bs=16, L~U[1024,8192]
  long_skew    4 seqs, 32 / 8,             D=128, bs=32, L={131072,512,512,512},
              split into 512-token context partitions

Conventions (all bf16 tensors are held as uint16 bit patterns):
  q            [S, Hq, D]
  k/v cache    [NB, Hkv, bs, D]     token t of seq i lives in block
                                    block_tables[i, t // bs] at offset t % bs
  block_tables [S, MB] int32        entries past ceil(L_i/bs) are poisoned
                                    (-1 or 0x7fffffff, alternating)
  context_lens [S] int32
  new_k/new_v  [T, Hkv, D]          tokens appended through slot_mapping [T] int64
Cache positions that hold no token (the tail of each sequence's last block,
blocks no table references, and the slot an append is about to fill) carry
the bf16 NaN 0x7FC0, so that any read that reaches the output shows up.
"""
from __future__ import annotations

import ctypes
import hashlib
import math
import os
import subprocess
from dataclasses import dataclass, field
from typing import Optional, Sequence

import numpy as np

BF16_NAN = 0x7FC0
TABLE_POISON = (-1, 0x7FFFFFFF)

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gen.c")
_LIB = None

# counter-based streams of the element generator
STREAM_Q, STREAM_K, STREAM_V, STREAM_NEW_K, STREAM_NEW_V = 1, 2, 3, 4, 5


def _lib_path() -> str:
    with open(_SRC, "rb") as f:
        digest = hashlib.sha256(f.read()).hexdigest()[:12]
    return os.path.join(_HERE, f"_libwlgen_{digest}.so")


def build_generator() -> str:
    """Compile gen.c with gcc (OpenMP when available); returns the .so path."""
    path = _lib_path()
    if os.path.exists(path):
        return path
    tmp = path + f".tmp{os.getpid()}"
    base = ["gcc", "-O2", "-shared", "-fPIC", "-std=c11", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)
    os.replace(tmp, path)
    return path


def _lib():
    global _LIB
    if _LIB is None:
        lib = ctypes.CDLL(build_generator())
        i64, u64 = ctypes.c_int64, ctypes.c_uint64
        lib.wl_normal_bf16.argtypes = [ctypes.c_void_p, i64, u64, u64, i64, ctypes.c_int]
        lib.wl_normal_bf16.restype = None
        lib.wl_u64.argtypes = [ctypes.c_void_p, i64, u64, u64, i64]
        lib.wl_u64.restype = None
        lib.wl_fill_u16.argtypes = [ctypes.c_void_p, i64, ctypes.c_uint16, ctypes.c_int]
        lib.wl_fill_u16.restype = None
        lib.wl_max_threads.argtypes = []
        lib.wl_max_threads.restype = ctypes.c_int
        _LIB = lib
    return _LIB


def normal_bf16(shape, seed: int, stream: int, offset: int = 0, threads: int = 0) -> np.ndarray:
    """bf16 bit patterns of approximately N(0,1) values, element j = draw(offset + j)."""
    out = np.empty(shape, dtype=np.uint16)
    _lib().wl_normal_bf16(out.ctypes.data, out.size, seed, stream, offset, threads)
    return out


def fill_u16(arr: np.ndarray, value: int, threads: int = 0) -> None:
    assert arr.dtype == np.uint16 and arr.flags.c_contiguous
    _lib().wl_fill_u16(arr.ctypes.data, arr.size, value, threads)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float32 (the bf16 is the top half)."""
    return (bits.astype(np.uint32) << np.uint32(16)).view(np.float32)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bf16 (nearest, ties to even); inputs must be finite."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = (u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))) >> np.uint64(16)
    return u.astype(np.uint16)


@dataclass
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    context_lens: np.ndarray          # [S] int32
    block_tables: np.ndarray          # [S, MB] int32
    q: np.ndarray                     # [S, Hq, D] uint16 (bf16 bits)
    k_cache: np.ndarray               # [NB, Hkv, bs, D] uint16, state before any append
    v_cache: np.ndarray
    scale: float
    seed: int
    new_k: Optional[np.ndarray] = None        # [T, Hkv, D] uint16
    new_v: Optional[np.ndarray] = None
    slot_mapping: Optional[np.ndarray] = None  # [T] int64
    partition_size: Optional[int] = None
    notes: dict = field(default_factory=dict)

    @property
    def max_blocks_per_seq(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_context_len(self) -> int:
        return int(self.context_lens.max()) if self.num_seqs else 0

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    def algorithmic_bytes(self, with_append: bool = False) -> int:
        """Bytes the decode step must move: valid K/V, q, fp32 out, table entries used, lengths."""
        L = self.context_lens.astype(np.int64)
        S, Hq, Hkv, D, bs = self.num_seqs, self.num_q_heads, self.num_kv_heads, self.head_dim, self.block_size
        b = int(L.sum()) * Hkv * D * 2 * 2 + S * Hq * D * 2 + S * Hq * D * 4
        b += int(((L + bs - 1) // bs).sum()) * 4 + S * 4
        if with_append and self.slot_mapping is not None:
            T = int(self.slot_mapping.shape[0])
            valid = int((self.slot_mapping >= 0).sum())
            b += T * 8 + T * Hkv * D * 2 * 2 + valid * Hkv * D * 2 * 2
        return b


def _lengths(kind, args, S, rng) -> np.ndarray:
    if kind == "fixed":
        L = np.asarray(args, dtype=np.int64)
        assert L.shape == (S,)
    elif kind == "uniform":       # integer-uniform, both ends included
        lo, hi = args
        L = rng.integers(lo, hi, size=S, endpoint=True)
    elif kind == "loguniform":    # round(exp(U(ln lo, ln hi))), clamped
        lo, hi = args
        L = np.rint(np.exp(rng.uniform(math.log(lo), math.log(hi), size=S))).astype(np.int64)
        L = np.clip(L, lo, hi)
    else:
        raise ValueError(kind)
    return L.astype(np.int32)


def make_workload(name: str, num_seqs: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  block_size: int, lengths, seed: int, pool: Optional[int] = None,
                  pool_scale: int = 1, append: bool = False, num_skip_slots: int = 0,
                  outlier_frac: float = 0.0, outlier_factor: int = 8,
                  partition_size: Optional[int] = None, threads: int = 0) -> Workload:
    """Build one seeded workload.

    `lengths` is ("fixed", [..]) / ("uniform", lo, hi) / ("loguniform", lo, hi) or a sequence.
    The numpy PCG64 stream is consumed in a fixed order: lengths, table permutation,
    key-outlier rows, slots that are skipped; q/k/v values come from the counter-based
    generator, indexed by their flat position, so they do not depend on that order.
    """
    S, Hq, Hkv, D, bs = num_seqs, num_q_heads, num_kv_heads, head_dim, block_size
    assert Hq % Hkv == 0
    rng = np.random.Generator(np.random.PCG64(seed))
    if isinstance(lengths, tuple) and isinstance(lengths[0], str):
        L = _lengths(lengths[0], lengths[1:] if lengths[0] != "fixed" else lengths[1], S, rng)
    else:
        L = np.asarray(lengths, dtype=np.int32)
        assert L.shape == (S,)
    nblk = (L.astype(np.int64) + bs - 1) // bs
    needed = int(nblk.sum())
    NB = pool if pool is not None else max(needed * pool_scale, 1)
    assert NB >= needed, "pool too small"
    MB = max(int(nblk.max()) if S else 0, 1)

    perm = rng.permutation(NB).astype(np.int32)
    tables = np.empty((S, MB), dtype=np.int32)
    poison = np.resize(np.asarray(TABLE_POISON, dtype=np.int64), MB).astype(np.int32)
    tables[:] = poison
    pos = 0
    for i in range(S):
        n = int(nblk[i])
        tables[i, :n] = perm[pos:pos + n]
        pos += n

    q = normal_bf16((S, Hq, D), seed, STREAM_Q, threads=threads)
    k_cache = normal_bf16((NB, Hkv, bs, D), seed, STREAM_K, threads=threads)
    v_cache = normal_bf16((NB, Hkv, bs, D), seed, STREAM_V, threads=threads)

    # poison every pool block that no table references ...
    used = np.zeros(NB, dtype=bool)
    used[perm[:needed]] = True
    unused = np.nonzero(~used)[0]
    if unused.size:
        k_cache[unused] = BF16_NAN
        v_cache[unused] = BF16_NAN
    # ... and the tail of each sequence's last block
    for i in range(S):
        tail = int(L[i]) % bs
        if nblk[i] and tail:
            b = tables[i, nblk[i] - 1]
            k_cache[b, :, tail:, :] = BF16_NAN
            v_cache[b, :, tail:, :] = BF16_NAN

    wl = Workload(name=name, num_seqs=S, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D,
                  block_size=bs, num_blocks=NB, context_lens=L, block_tables=tables, q=q,
                  k_cache=k_cache, v_cache=v_cache, scale=1.0 / math.sqrt(D), seed=seed,
                  partition_size=partition_size)

    if outlier_frac > 0:
        # whole key rows (one token, one kv head) scaled by 8: exact in bf16
        rows = rng.random((NB, Hkv, bs)) < outlier_frac
        k_cache[rows] = _times_pow2(k_cache[rows], outlier_factor)
        wl.notes["outlier_rows_cache"] = int(rows.sum())

    if append:
        T = S
        new_k = normal_bf16((T, Hkv, D), seed, STREAM_NEW_K, threads=threads)
        new_v = normal_bf16((T, Hkv, D), seed, STREAM_NEW_V, threads=threads)
        if outlier_frac > 0:
            rows = rng.random((T, Hkv)) < outlier_frac
            new_k[rows] = _times_pow2(new_k[rows], outlier_factor)
        skip = np.zeros(T, dtype=bool)
        if num_skip_slots:
            skip[rng.choice(T, size=num_skip_slots, replace=False)] = True
        slots = np.full(T, -1, dtype=np.int64)
        for i in range(S):
            t = int(L[i]) - 1
            if skip[i] or t < 0:
                continue
            b = int(tables[i, t // bs])
            slots[i] = b * bs + t % bs
            # the slot the append fills holds no token yet
            k_cache[b, :, t % bs, :] = BF16_NAN
            v_cache[b, :, t % bs, :] = BF16_NAN
        wl.new_k, wl.new_v, wl.slot_mapping = new_k, new_v, slots
    return wl


STREAM_MULTI_Q = 6


def multi_query(wl: Workload, q_len: int, threads: int = 0) -> np.ndarray:
    """Queries of q_len new tokens per sequence, [S, q_len, Hq, D] bf16 bits (the tokens
    themselves are the last q_len positions already in the workload's cache)."""
    return normal_bf16((wl.num_seqs, q_len, wl.num_q_heads, wl.head_dim), wl.seed, STREAM_MULTI_Q, threads=threads)


def _times_pow2(bits: np.ndarray, factor: int) -> np.ndarray:
    x = bf16_bits_to_f32(bits) * np.float32(factor)
    return f32_to_bf16_bits(x)


@dataclass(frozen=True)
class ConfigSpec:
    index: int
    name: str
    kwargs: dict
    description: str


CONFIGS = {
    1: ConfigSpec(1, "tiny", dict(num_seqs=4, num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                                  lengths=("fixed", [1, 17, 33, 64]), pool=32, seed=0),
                  "tiny paged decode: 4 seqs, 4 q / 2 kv heads, D=64, bs=16, L={1,17,33,64}, 32-block pool"),
    2: ConfigSpec(2, "tinyllama", dict(num_seqs=8, num_q_heads=32, num_kv_heads=4, head_dim=64, block_size=16,
                                       lengths=("uniform", 128, 2048), pool_scale=2, seed=2),
                  "TinyLlama-1.1B-shaped layer: 8 seqs, 32 q / 4 kv heads, D=64, bs=16, L~U[128,2048], pool 2x"),
    3: ConfigSpec(3, "cont_batch", dict(num_seqs=64, num_q_heads=32, num_kv_heads=32, head_dim=128,
                                        block_size=16, lengths=("loguniform", 16, 4096), seed=3, append=True,
                                        num_skip_slots=8, outlier_frac=0.01),
                  "continuous-batch mix: 64 seqs, 32/32 heads (MHA), D=128, bs=16, L~logU[16,4096], "
                  "1 appended token per seq (8 slots=-1), 1% key rows x8"),
    4: ConfigSpec(4, "llama3_8b", dict(num_seqs=256, num_q_heads=32, num_kv_heads=8, head_dim=128,
                                       block_size=16, lengths=("uniform", 1024, 8192), seed=4),
                  "Llama-3-8B-shaped GQA decode: 256 seqs, 32 q / 8 kv heads, D=128, bs=16, L~U[1024,8192]"),
    5: ConfigSpec(5, "long_skew", dict(num_seqs=4, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=32,
                                       lengths=("fixed", [131072, 512, 512, 512]), seed=5, partition_size=512),
                  "long-context skew: 4 seqs, 32 q / 8 kv heads, D=128, bs=32, L={131072,512,512,512}, "
                  "512-token partitions"),
}


def make_config(index: int, threads: int = 0) -> Workload:
    spec = CONFIGS[index]
    return make_workload(spec.name, threads=threads, **spec.kwargs)


def seed_all_lengths(index: int) -> np.ndarray:
    """The context lengths of a named workload without generating its tensors."""
    spec = CONFIGS[index]
    kw = spec.kwargs
    rng = np.random.Generator(np.random.PCG64(kw["seed"]))
    lk = kw["lengths"]
    return _lengths(lk[0], lk[1:] if lk[0] != "fixed" else lk[1], kw["num_seqs"], rng)


__all__ = ["Workload", "CONFIGS", "make_config", "make_workload", "normal_bf16", "bf16_bits_to_f32",
           "f32_to_bf16_bits", "fill_u16", "seed_all_lengths", "BF16_NAN",
           "build_generator"]
