"""Microbenchmarks of the GB300 units behind the sparse path's kernel choices.

    python bench_micro.py [gather] [churn] [stream] [tma_ring] [mma] [umma] [cvt] [sf_layout]   (default: all)

Prints one JSON line per measurement (CUDA events on the launching stream,
best of 5 after a warm-up).  See bench_micro.cu for what each one runs:
  gather     GB/s of a 4 KB page-pair gather by 1-D TMA into shared memory,
             from a pool that fits L2 (16..128 MB) or does not (1 GB): the
             data-movement ceiling of an attention over selected pages
  churn      the same HBM gather with the bytes spread over many short CTAs
             (4..128 pages each): what a CTA's start and end cost in
             bandwidth
  stream     GB/s of read-only streams over a 4 GB pool, every byte read
             once (nothing for L2 to serve): plain 16-byte loads, the page
             gather above on a permutation, and whole 16896-byte chunks (an
             fp8 index field) through a CTA ring of 1, 2 or 4 stages
  tma_ring   bytes per SM clock of the fp8 prefill scorer's key loads alone
             (two 16 KB boxes a tile, a 4- or 6-stage ring, one CTA per SM)
             from a pool that fits L2 (32 MB) or not (2 GB): 2-D tensor loads
             with 128-byte swizzle against 1-D bulk copies
  mma        TFLOP/s of mma.sync m16n8k16 f16 and m16n8k32 e4m3
  umma       TFLOP/s of tcgen05.mma (one issuing thread, M = 128) by N, and
             with N = 16 into several independent accumulators
  cvt        e4m3x2 -> f16x2 conversions per clock per SM
  sf_layout  checks where kind::mxf8f6f4.block_scale reads its scale
             factors in TMEM: row r's cell at lanes 32p + r % 32 of every
             sub-partition p, column base + r / 32 (the MXFP4 prefill scorer
             relies on it)
"""
import ctypes as C
import json
import os
import subprocess
import sys

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
LIB = os.path.join(ROOT, "_build", "libbench_micro.so")


def build():
    os.makedirs(os.path.dirname(LIB), exist_ok=True)
    src = os.path.join(ROOT, "bench_micro.cu")
    if os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(src):
        return LIB
    subprocess.check_call(["nvcc", "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-lineinfo", "-std=c++17",
                           "-Xcompiler", "-fPIC", "--expt-relaxed-constexpr", "-shared", "-I", ROOT, "-I",
                           os.path.join(ROOT, "include"), src,
                           "-o", LIB, "-lcuda"])
    return LIB


def main():
    which = [a for a in sys.argv[1:] if not a.startswith("-")] or ["gather", "churn", "stream", "tma_ring", "mma",
                                                                    "umma", "cvt", "sf_layout"]
    L = C.CDLL(build())
    vp, i32 = C.c_void_p, C.c_int
    L.micro_gather.argtypes = [vp, vp, i32, i32, i32, vp, vp, vp]
    L.micro_mma_sync.argtypes = [i32, i32, vp, i32, vp]
    L.micro_stream_ld.argtypes = [vp, C.c_int64, i32, vp, vp]
    L.micro_chunk.argtypes = [vp, vp, i32, i32, i32, i32, vp, vp, vp]
    L.micro_tma_ring.argtypes = [vp, C.c_int64, vp, i32, i32, i32, i32, vp, vp, vp]
    L.micro_umma.argtypes = [i32, i32, i32, i32, vp, vp, vp]
    L.micro_umma_multi.argtypes = [i32, i32, i32, vp, vp, vp]
    L.micro_cvt.argtypes = [i32, i32, vp, vp]
    L.micro_sf_layout.argtypes = [vp, vp, i32, i32, vp, vp, vp]
    dev = "cuda"
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    s = torch.cuda.current_stream()
    sp = C.c_void_p(s.cuda_stream)
    err = torch.zeros(1, dtype=torch.int32, device=dev)

    def timed(fn, reps=5):
        assert fn() == 0
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(s)
            fn()
            b.record(s)
            torch.cuda.synchronize()
            ts.append(a.elapsed_time(b))
        return min(ts)

    def emit(d):
        print(json.dumps(d), flush=True)

    if "gather" in which:
        rng = np.random.default_rng(0)
        for nblocks, rows in ((512, 16384), (4096, 16384), (32768, 16384), (32768, 512)):
            pool = torch.zeros(nblocks * 32768, dtype=torch.uint8, device=dev)
            # page ids of an interleaved fp8 cache: block*16 + j, j < 8 (K page; V 8 slots on)
            ids = torch.from_numpy((rng.integers(0, nblocks, (rows, 128)) * 16 +
                                    rng.integers(0, 8, (rows, 128))).astype(np.int32)).to(dev)
            sink = torch.zeros(rows * 128, dtype=torch.int32, device=dev)
            for ring in (2, 3, 4):
                ms = timed(lambda: L.micro_gather(pool.data_ptr(), ids.data_ptr(), rows, 128, ring, sink.data_ptr(),
                                                  err.data_ptr(), sp))
                emit({"micro": "gather", "pool_MB": nblocks * 32768 / 2 ** 20, "rows": rows, "pages_per_row": 128,
                      "ring": ring, "ms": ms, "GB_per_s": rows * 128 * 4096 / (ms / 1e3) / 1e9})
            del pool
    if "churn" in which:  # the same bytes from HBM by many short CTAs instead of fewer long ones
        rng = np.random.default_rng(1)
        nblocks = 32768
        pool = torch.zeros(nblocks * 32768, dtype=torch.uint8, device=dev)
        for rows, ppr in ((16384, 128), (65536, 32), (262144, 8), (524288, 4)):
            ids = torch.from_numpy((rng.integers(0, nblocks, (rows, ppr)) * 16 +
                                    rng.integers(0, 8, (rows, ppr))).astype(np.int32)).to(dev)
            sink = torch.zeros(rows * 128, dtype=torch.int32, device=dev)
            for ring in (2,):
                ms = timed(lambda: L.micro_gather(pool.data_ptr(), ids.data_ptr(), rows, ppr, ring, sink.data_ptr(),
                                                  err.data_ptr(), sp))
                emit({"micro": "gather_churn", "pool_MB": nblocks * 32768 / 2 ** 20, "rows": rows,
                      "pages_per_row": ppr, "ring": ring, "ms": ms, "GB_per_s": rows * ppr * 4096 / (ms / 1e3) / 1e9})
        del pool
    if "stream" in which:  # every byte of a 4 GB pool read once
        rng = np.random.default_rng(2)
        pool_bytes = 4 << 30
        pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
        sink = torch.zeros(sms * 32 * 256, dtype=torch.int32, device=dev)
        for per_sm in (4, 8, 16, 32):
            ms = timed(lambda: L.micro_stream_ld(pool.data_ptr(), pool_bytes, sms * per_sm, sink.data_ptr(), sp))
            emit({"micro": "stream_ld", "pool_MB": pool_bytes >> 20, "ctas_per_sm": per_sm, "threads": 256,
                  "ms": ms, "GB_per_s": pool_bytes / (ms / 1e3) / 1e9})
        # page pairs (block * 16 + j, j < 8, and its partner 8 slots on) in a random order, each once
        nblk = pool_bytes // 32768
        ids = torch.from_numpy(rng.permutation(nblk * 8).astype(np.int64)).to(dev)
        ids = (ids // 8 * 16 + ids % 8).to(torch.int32)
        rows = nblk * 8 // 128
        gsink = torch.zeros(rows * 128, dtype=torch.int32, device=dev)
        for ring in (2, 4):
            ms = timed(lambda: L.micro_gather(pool.data_ptr(), ids.data_ptr(), rows, 128, ring, gsink.data_ptr(),
                                              err.data_ptr(), sp))
            emit({"micro": "stream_gather", "pool_MB": pool_bytes >> 20, "rows": rows, "pages_per_row": 128,
                  "ring": ring, "ms": ms, "GB_per_s": rows * 128 * 4096 / (ms / 1e3) / 1e9})
        del ids, gsink
        chunk = 16896
        nchunk = pool_bytes // chunk
        perm = torch.from_numpy(rng.permutation(nchunk).astype(np.int32)).to(dev)
        for cpc in (2, 4, 16):
            ctas = nchunk // cpc
            csink = torch.zeros(ctas * 128, dtype=torch.int32, device=dev)
            for st in (1, 2, 4):
                ms = timed(lambda: L.micro_chunk(pool.data_ptr(), perm.data_ptr(), ctas, cpc, chunk, st,
                                                 csink.data_ptr(), err.data_ptr(), sp))
                emit({"micro": "stream_chunk", "chunk_bytes": chunk, "chunks_per_cta": cpc, "stages": st,
                      "ctas": ctas, "ms": ms, "GB_per_s": ctas * cpc * chunk / (ms / 1e3) / 1e9})
        del pool, perm
    if "tma_ring" in which:  # the prefill scorer's key loads alone
        rng = np.random.default_rng(4)
        clk = 2.07e9
        for pool_bytes in (32 << 20, 2 << 30):
            pool = torch.zeros(pool_bytes, dtype=torch.uint8, device=dev)
            blocks = pool_bytes // 16896
            tiles = 256
            # block b's keys start at row b * 132 (16896-byte fields seen as 128-byte rows)
            rows = torch.from_numpy((rng.integers(0, blocks - 1, (sms, tiles * 2)) * 132).astype(np.int32)).to(dev)
            tsink = torch.zeros(sms, dtype=torch.int32, device=dev)
            for st in (4, 6):
                for mode in (0, 1):
                    ms = timed(lambda: L.micro_tma_ring(pool.data_ptr(), pool_bytes, rows.data_ptr(), sms, tiles, st,
                                                        mode, tsink.data_ptr(), err.data_ptr(), sp))
                    b = sms * tiles * 32768
                    emit({"micro": "tma_ring", "pool_MB": pool_bytes >> 20, "stages": st,
                          "copy": "2-D tensor, 128B swizzle" if mode == 0 else "1-D bulk",
                          "ms": ms, "GB_per_s": b / (ms / 1e3) / 1e9,
                          "bytes_per_sm_clock_at_2.07GHz": b / sms / (ms / 1e3) / clk})
            del pool
    if "mma" in which:
        out = torch.zeros(sms * 8 * 256, dtype=torch.float32, device=dev)
        for e4m3 in (0, 1):
            for cps in (2, 4, 8):
                iters = 4000
                ms = timed(lambda: L.micro_mma_sync(sms * cps, iters, out.data_ptr(), e4m3, sp))
                flop = sms * cps * 8 * iters * 8 * (2 * 16 * 8 * (32 if e4m3 else 16))
                emit({"micro": "mma_sync", "shape": "m16n8k32.e4m3" if e4m3 else "m16n8k16.f16",
                      "warps_per_sm": cps * 8, "ms": ms, "TFLOP_per_s": flop / (ms / 1e3) / 1e12})
    if "umma" in which:
        sink = torch.zeros(sms * 128, dtype=torch.int32, device=dev)
        for kind in (0, 1):
            for n in (16, 32, 64, 128, 256):
                iters = 20000 if n <= 64 else 5000
                ms = timed(lambda: L.micro_umma(sms, iters, n, kind, err.data_ptr(), sink.data_ptr(), sp))
                k = 16 if kind == 0 else 32
                emit({"micro": "umma", "kind": "f16" if kind == 0 else "f8f6f4.e4m3", "M": 128, "N": n, "K": k,
                      "ms": ms, "TFLOP_per_s": sms * iters * 2 * 128 * n * k / (ms / 1e3) / 1e12,
                      "ns_per_mma": ms * 1e6 / iters})
        for nacc in (1, 2, 4, 8, 16):
            iters = 32000
            ms = timed(lambda: L.micro_umma_multi(sms, iters, nacc, err.data_ptr(), sink.data_ptr(), sp))
            emit({"micro": "umma_accumulators", "kind": "f16", "M": 128, "N": 16, "K": 16, "accumulators": nacc,
                  "ms": ms, "TFLOP_per_s": sms * iters * 2 * 128 * 16 * 16 / (ms / 1e3) / 1e12,
                  "ns_per_mma": ms * 1e6 / iters})
    if "cvt" in which:
        out = torch.zeros(sms * 8 * 256, dtype=torch.int32, device=dev)
        for cps in (2, 4, 8):
            iters = 4000
            ms = timed(lambda: L.micro_cvt(sms * cps, iters, out.data_ptr(), sp))
            n = sms * cps * 256 * iters * 8
            emit({"micro": "cvt.rn.f16x2.e4m3x2", "threads_per_sm": cps * 256, "ms": ms,
                  "per_ns_per_sm": n / (ms * 1e6) / sms})
    if "sf_layout" in which:
        rng = np.random.default_rng(3)
        xa = rng.integers(120, 135, (128, 4)).astype(np.uint8)
        xb = rng.integers(120, 135, (128, 4)).astype(np.uint8)
        ta = np.zeros((128, 8, 4), np.uint8)
        tb = np.zeros((128, 8, 4), np.uint8)
        for p in range(4):
            for r in range(128):
                ta[32 * p + r % 32, r // 32] = xa[r]
                tb[32 * p + r % 32, r // 32] = xb[r]
        sa = torch.from_numpy(ta.view(np.uint32).reshape(-1).copy()).to(dev)
        sb = torch.from_numpy(tb.view(np.uint32).reshape(-1).copy()).to(dev)
        out = torch.zeros(128 * 128, dtype=torch.float32, device=dev)
        for a_id, b_id in ((0, 0), (1, 2), (3, 1), (2, 3)):
            assert L.micro_sf_layout(sa.data_ptr(), sb.data_ptr(), a_id, b_id, out.data_ptr(), err.data_ptr(), sp) == 0
            torch.cuda.synchronize()
            d = out.cpu().numpy().reshape(128, 128)
            h = 32.0 * np.exp2(xa[:, a_id].astype(np.float64) - 127)[:, None] * \
                np.exp2(xb[:, b_id].astype(np.float64) - 127)[None, :]
            emit({"micro": "sf_layout", "a_sf_id": a_id, "b_sf_id": b_id, "layout_matches": bool(np.array_equal(d, h))})
    torch.cuda.synchronize()
    emit({"micro": "device_errors", "value": int(err.item())})


if __name__ == "__main__":
    main()
