"""CPU oracle for paged-KV decode attention -- TEST INFRASTRUCTURE.

Only `tests/`, `__graft_entry__.smoke()` and the bench's CPU-baseline /
reference leg may import this package.  The product library
(`paged_kv_decode_pf_gb300`) never imports it and shares no code with it.

`pf_oracle.c` is the fp64 restatement of the method (KV append, paged decode
attention with grouped-query heads, split over context partitions with a
log-sum-exp merge); `dense.py` is a pure-Python brute force over contiguous
K/V that pins it.  This module compiles the C file with gcc and exposes it on
numpy arrays; inputs are bf16 bit patterns held as uint16.

Parity pins (all in tests/test_oracle_pins.py): brute-force dense attention,
a torch float64 library witness, block-permutation invariance, L=1, equal
keys / q=0 / scale=0, constant V, a dominant key, GQA == MHA with repeated kv
heads, split == unsplit for several partition sizes, a bit-exact numpy scatter
for the append, and mutants of this file that those pins must reject.
"""
from __future__ import annotations

import ctypes
import hashlib
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pf_oracle.c")
_LIB = None


def compile_oracle(source: str = SOURCE, out_dir: Optional[str] = None, openmp: bool = True) -> str:
    """gcc-compile an oracle source into a shared object named after its content hash."""
    with open(source, "rb") as f:
        text = f.read()
    digest = hashlib.sha256(text + (b"omp" if openmp else b"")).hexdigest()[:12]
    out_dir = out_dir or _HERE
    path = os.path.join(out_dir, f"_liboracle_{digest}.so")
    if os.path.exists(path):
        return path
    tmp = path + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-shared", "-fPIC", source, "-o", tmp, "-lm"]
    if openmp:
        try:
            subprocess.run(cmd[:1] + ["-fopenmp"] + cmd[1:], check=True, capture_output=True)
        except subprocess.CalledProcessError:
            subprocess.run(cmd, check=True, capture_output=True)
    else:
        subprocess.run(cmd, check=True, capture_output=True)
    os.replace(tmp, path)
    return path


def _bind(lib):
    P, i32, i64, f64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
    lib.oracle_reshape_and_cache.argtypes = [P, P, P, P, P, i64, i32, i32, i32, i64]
    lib.oracle_reshape_and_cache.restype = i64
    lib.oracle_paged_attention.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64, P, i32]
    lib.oracle_paged_attention.restype = None
    lib.oracle_paged_attention_partition.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, f64,
                                                     i32, i32, P, P, P, i32]
    lib.oracle_paged_attention_partition.restype = None
    lib.oracle_merge.argtypes = [P, P, P, P, i32, i32, i32, i32, i32, P]
    lib.oracle_merge.restype = None
    lib.oracle_max_threads.argtypes = []
    lib.oracle_max_threads.restype = i32
    lib.oracle_copy_blocks.argtypes = [P, P, P, i64, i32, i32, i32, i64]
    lib.oracle_copy_blocks.restype = i64
    lib.oracle_paged_attention_multi.argtypes = [P, P, P, P, P, i32, i32, i32, i32, i32, i32, i32, f64, P, i32]
    lib.oracle_paged_attention_multi.restype = None
    return lib


def load(path: Optional[str] = None):
    """The compiled oracle (the default source unless `path` names another .so)."""
    global _LIB
    if path is not None:
        return Oracle(_bind(ctypes.CDLL(path)))
    if _LIB is None:
        _LIB = Oracle(_bind(ctypes.CDLL(compile_oracle())))
    return _LIB


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data


class Oracle:
    """numpy front end of one compiled oracle shared object."""

    def __init__(self, lib):
        self.lib = lib

    def max_threads(self) -> int:
        return int(self.lib.oracle_max_threads())

    def reshape_and_cache(self, k, v, slot_mapping, k_cache, v_cache, block_size):
        """Returns new (k_cache, v_cache) copies and the count of out-of-range slots."""
        T, Hkv, D = k.shape
        NB = k_cache.shape[0]
        kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16, copy=True)
        k, kp = _c(k, np.uint16)
        v, vp = _c(v, np.uint16)
        s, sp = _c(slot_mapping, np.int64)
        bad = self.lib.oracle_reshape_and_cache(kp, vp, sp, kc.ctypes.data, vc.ctypes.data, T, Hkv, D,
                                                block_size, NB)
        return kc, vc, int(bad)

    def copy_blocks(self, k_cache, v_cache, block_mapping):
        """Returns new (k_cache, v_cache) after copying block_mapping[j] = (src, dst) pairs, and the
        count of pairs skipped for an out-of-range id."""
        NB, Hkv, bs, D = k_cache.shape
        kc, vc = np.array(k_cache, dtype=np.uint16, copy=True), np.array(v_cache, dtype=np.uint16, copy=True)
        bm, bp = _c(np.asarray(block_mapping).reshape(-1, 2), np.int64)
        bad = self.lib.oracle_copy_blocks(kc.ctypes.data, vc.ctypes.data, bp, bm.shape[0], Hkv, D, bs, NB)
        return kc, vc, int(bad)

    def paged_attention(self, q, k_cache, v_cache, block_tables, context_lens, scale, threads: int = 0):
        S, Hq, D = q.shape
        NB, Hkv, bs, D2 = k_cache.shape
        assert D == D2
        q, qp = _c(q, np.uint16)
        kc, kp = _c(k_cache, np.uint16)
        vc, vp = _c(v_cache, np.uint16)
        bt, bp = _c(block_tables, np.int32)
        cl, cp = _c(context_lens, np.int32)
        out = np.zeros((S, Hq, D), dtype=np.float64)
        self.lib.oracle_paged_attention(qp, kp, vp, bp, cp, S, Hq, Hkv, D, bs, bt.shape[1], float(scale),
                                        out.ctypes.data, threads)
        return out

    def paged_attention_multi(self, q, k_cache, v_cache, block_tables, context_lens, scale, threads: int = 0):
        """q [S, q_len, Hq, D] -> out [S, q_len, Hq, D]; row (i, j) sees tokens t <= L_i - q_len + j."""
        S, Q, Hq, D = q.shape
        NB, Hkv, bs, _ = k_cache.shape
        q, qp = _c(q, np.uint16)
        kc, kp = _c(k_cache, np.uint16)
        vc, vp = _c(v_cache, np.uint16)
        bt, bp = _c(block_tables, np.int32)
        cl, cp = _c(context_lens, np.int32)
        out = np.zeros((S, Q, Hq, D), dtype=np.float64)
        self.lib.oracle_paged_attention_multi(qp, kp, vp, bp, cp, S, Q, Hq, Hkv, D, bs, bt.shape[1], float(scale),
                                              out.ctypes.data, threads)
        return out

    def partition(self, q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                  max_partitions=None, threads: int = 0):
        S, Hq, D = q.shape
        NB, Hkv, bs, _ = k_cache.shape
        cl = np.ascontiguousarray(context_lens, dtype=np.int32)
        if max_partitions is None:
            mx = int(cl.max()) if S else 0
            max_partitions = max((mx + partition_size - 1) // partition_size, 1)
        q, qp = _c(q, np.uint16)
        kc, kp = _c(k_cache, np.uint16)
        vc, vp = _c(v_cache, np.uint16)
        bt, bp = _c(block_tables, np.int32)
        o = np.zeros((S, Hq, max_partitions, D), dtype=np.float64)
        m = np.zeros((S, Hq, max_partitions), dtype=np.float64)
        l = np.zeros((S, Hq, max_partitions), dtype=np.float64)
        self.lib.oracle_paged_attention_partition(qp, kp, vp, bp, cl.ctypes.data, S, Hq, Hkv, D, bs,
                                                  bt.shape[1], float(scale), partition_size, max_partitions,
                                                  o.ctypes.data, m.ctypes.data, l.ctypes.data, threads)
        return o, m, l

    def merge(self, tmp_out, tmp_m, tmp_l, context_lens, partition_size):
        S, Hq, NP, D = tmp_out.shape
        o, op = _c(tmp_out, np.float64)
        m, mp = _c(tmp_m, np.float64)
        l, lp = _c(tmp_l, np.float64)
        cl, cp = _c(context_lens, np.int32)
        out = np.zeros((S, Hq, D), dtype=np.float64)
        self.lib.oracle_merge(op, mp, lp, cp, S, Hq, D, partition_size, NP, out.ctypes.data)
        return out

    def split_attention(self, q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                        threads: int = 0):
        o, m, l = self.partition(q, k_cache, v_cache, block_tables, context_lens, scale, partition_size,
                                 threads=threads)
        return self.merge(o, m, l, context_lens, partition_size)
