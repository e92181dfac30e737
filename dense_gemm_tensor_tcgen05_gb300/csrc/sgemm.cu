// sgemm.cu -- CUDA-core kernels: the FP32 SGEMM, a guarded generic GEMM for
// inputs the vectorised or TMA paths cannot take, and the K == 0 fill.
//
// SGEMM design (the register-tiling ladder of "matmul_registers.cu" carried
// to its last step, re-derived for sm_103a):
//   * a CTA computes a BM x BN tile of C; each thread owns an 8 x 8 register
//     micro-tile split into four 4 x 4 quadrants (rows ty*4.. and BM/2+ty*4..,
//     columns tx*4.. and BN/2+tx*4..), so every shared-memory fragment read is
//     one float4 and a warp's reads hit distinct banks.  The wide form gives
//     each thread 8 x 16 outputs (column chunks tx*4.. + c*BN/4): 128 FMAs per
//     6 float4 shared loads, at 128 threads per 128 x 128 tile;
//   * per K step of BK, A (BM x BK) and B (BK x BN) slices come in with float4
//     global loads; A is stored transposed (k-major rows of BM floats, padded
//     by 4 so the transposing stores are conflict-free), which makes the
//     inner loop read four consecutive rows of A with one instruction;
//   * two shared-memory buffers: the next slice is loaded into registers
//     while the current one is multiplied, then stored to the other buffer,
//     with one barrier per K step;
//   * 64 FMAs per 4 float4 shared loads in the inner loop, issued as 32
//     packed fma.rn.f32x2 (two FP32 FMAs per instruction).
// Edges: each CTA decides once whether its tile lies wholly inside C; only
// boundary tiles use guarded loads and masked stores, and only the last,
// partial K step of any tile uses guarded loads.  Misaligned pointers or
// leading dimensions go to the generic kernel instead.
// Schedules: one CTA per (tile, K slice), or stream-K -- a grid of exactly
// the CTAs that fit on the GPU at once, which first takes whole tiles while
// whole waves of them last and then shares the remaining tiles' K steps out
// evenly, so every SM does the same number of FMAs.  A tile cut into pieces
// is summed by its last piece to finish, in piece order.

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdio>

#include "cstore.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

// ---------------------------------------------------------------- SGEMM --

#ifndef GB300_SGEMM_BK
#define GB300_SGEMM_BK 16
#endif
constexpr int kSgemmBK = GB300_SGEMM_BK;

// One SGEMM configuration: a BM x BN CTA tile, K steps of BK, 8 x TN outputs
// per thread (TN = 8 or 16).  Shared memory holds two slices (double
// buffer); A is stored transposed, k-major rows of BM + 4 floats.  A
// thread's rows are ty*4.. and BM/2 + ty*4.., its columns TN/4 chunks of 4:
// c*BN/(TN/4) + tx*4.
template <int BM_, int BN_, int BK_, int TN_>
struct SgemmCfg {
    static constexpr int BM = BM_, BN = BN_, BK = BK_, TN = TN_;
    static constexpr int kTx = BN / TN;            // threads along N
    static constexpr int kTy = BM / 8;             // threads along M
    static constexpr int kThreads = kTx * kTy;
    static constexpr int kChunks = TN / 4;         // 4-wide column chunks per thread
    static constexpr int kAStride = BM + 4;        // padded row of the transposed A slice
    static constexpr int kAFloats = BK * kAStride; // one A slice
    static constexpr int kBFloats = BK * BN;       // one B slice
    static constexpr int kSmemBytes = 2 * (kAFloats + kBFloats) * 4;
    static constexpr int kALoads = BM * BK / 4;    // float4 per A slice
    static constexpr int kBLoads = BK * BN / 4;    // float4 per B slice
    static constexpr int kAPer = kALoads / kThreads;
    static constexpr int kBPer = kBLoads / kThreads;
    // resident CTAs per SM the register allocation must allow: 128 x 128 runs
    // 2, 128 x 64 runs 3 (4 warps each, <= 170 registers)
    static constexpr int kMinBlocks = (BM * BN >= 128 * 128) ? 2 : (BM * BN >= 128 * 64) ? 3 : 1;
    static_assert(TN == 8 || TN == 16, "micro-tile width");
    static_assert(BM % 8 == 0 && BN % TN == 0 && BK % 4 == 0, "tile shape");
    static_assert(kThreads % 32 == 0 && kThreads <= 1024, "whole warps");
    static_assert(kALoads % kThreads == 0 && kBLoads % kThreads == 0, "even load split");
    static_assert(kAFloats % 4 == 0, "16-byte aligned buffers");

    __device__ static __forceinline__ int row(int ty, int i) { return (i >> 2) * (BM / 2) + ty * 4 + (i & 3); }
    __device__ static __forceinline__ int col(int tx, int c) { return c * (BN / kChunks) + tx * 4; }
};

struct SgArgs {
    const float* A;
    const float* B;
    void* C;            // element type ct
    int M, N, K;
    int64_t lda, ldb, ldc;
    int tiles_n;        // tiles along N
    int tile0;          // first (row-major linear) tile of this launch
    int splits;         // K slices per tile; 1 = the whole K
    int k_chunk;        // K per slice, a multiple of BK
    int ab;             // 0: C = AB; 1: alpha AB; 2: alpha AB + beta C
    float alpha, beta;
    int ct;             // C's type (cstore.cuh)
    float* ws;          // split-K partial tiles of this launch
    uint32_t* counters; // split-K arrival counter per tile, zero between launches
    int sk_mode;        // 1: stream-K schedule (persistent grid)
    int dp_tiles;       // stream-K: tiles done whole, tile cta, cta + grid, ...
    int kb_total;       // stream-K: K steps (of BK) per tile
    int64_t sk_iters;   // stream-K: K steps shared out over the grid after dp_tiles
    int max_seg;        // stream-K: workspace slots per cut tile
};

// Packed FP32 pairs: fma.rn.f32x2 performs two independent single-rounding
// FMAs, the same arithmetic as two fmaf, in one instruction -- half the
// issue slots of the inner loop, which is what bounds this kernel.
__device__ __forceinline__ uint64_t f32x2_pack(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ void f32x2_unpack(uint64_t v, float& lo, float& hi) {
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}

__device__ __forceinline__ void f32x2_fma(uint64_t& acc, uint64_t a, uint64_t b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(acc) : "l"(a), "l"(b));
}

// Load one BK slice of A (BM x BK) and B (BK x BN) starting at k0 into
// registers.  Elements at k >= kend, or outside M / N in an edge tile, read
// as zero.
template <class Cfg, bool EDGE>
__device__ __forceinline__ void sgemm_load(const SgArgs& a, int m0, int n0, int k0, int kend,
                                           bool guard_k, float4 (&ra)[Cfg::kAPer],
                                           float4 (&rb)[Cfg::kBPer]) {
    constexpr int BK = Cfg::BK, BN = Cfg::BN;
    const int tid = threadIdx.x;
#pragma unroll
    for (int l = 0; l < Cfg::kAPer; ++l) {
        const int idx = tid + l * Cfg::kThreads;
        const int r = idx / (BK / 4);
        const int kq = (idx % (BK / 4)) * 4;
        const int gm = m0 + r, gk = k0 + kq;
        const float* src = a.A + static_cast<int64_t>(gm) * a.lda + gk;
        if (!EDGE && !guard_k) {
            ra[l] = __ldg(reinterpret_cast<const float4*>(src));
        } else if (gm < a.M && gk + 3 < kend) {
            ra[l] = __ldg(reinterpret_cast<const float4*>(src));
        } else {
            float t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) t[i] = (gm < a.M && gk + i < kend) ? __ldg(src + i) : 0.0f;
            ra[l] = make_float4(t[0], t[1], t[2], t[3]);
        }
    }
#pragma unroll
    for (int l = 0; l < Cfg::kBPer; ++l) {
        const int idx = tid + l * Cfg::kThreads;
        const int kr = idx / (BN / 4);
        const int nq = (idx % (BN / 4)) * 4;
        const int gk = k0 + kr, gn = n0 + nq;
        const float* src = a.B + static_cast<int64_t>(gk) * a.ldb + gn;
        if (!EDGE && !guard_k) {
            rb[l] = __ldg(reinterpret_cast<const float4*>(src));
        } else if (gk < kend && gn + 3 < a.N) {
            rb[l] = __ldg(reinterpret_cast<const float4*>(src));
        } else {
            float t[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) t[i] = (gk < kend && gn + i < a.N) ? __ldg(src + i) : 0.0f;
            rb[l] = make_float4(t[0], t[1], t[2], t[3]);
        }
    }
}

template <class Cfg>
__device__ __forceinline__ void sgemm_store_smem(float* As, float* Bs, const float4 (&ra)[Cfg::kAPer],
                                                 const float4 (&rb)[Cfg::kBPer]) {
    constexpr int BK = Cfg::BK, BN = Cfg::BN;
    const int tid = threadIdx.x;
#pragma unroll
    for (int l = 0; l < Cfg::kAPer; ++l) {
        const int idx = tid + l * Cfg::kThreads;
        const int r = idx / (BK / 4);
        const int kq = (idx % (BK / 4)) * 4;
        As[(kq + 0) * Cfg::kAStride + r] = ra[l].x;
        As[(kq + 1) * Cfg::kAStride + r] = ra[l].y;
        As[(kq + 2) * Cfg::kAStride + r] = ra[l].z;
        As[(kq + 3) * Cfg::kAStride + r] = ra[l].w;
    }
#pragma unroll
    for (int l = 0; l < Cfg::kBPer; ++l) {
        const int idx = tid + l * Cfg::kThreads;
        const int kr = idx / (BN / 4);
        const int nq = (idx % (BN / 4)) * 4;
        *reinterpret_cast<float4*>(Bs + kr * BN + nq) = rb[l];
    }
}

// acc2 (this thread's outputs as column pairs) += one BK slice from shared
// memory.  With PF the fragments of step k + 1 are read before the FMAs of
// step k (two register sets); without it each step reads its own.  PF
// measured 1-7 % faster for the split kernel's whole tiles and 2-4 % slower
// for the stream-K form, which uses it off.
template <class Cfg, bool PF>
__device__ __forceinline__ void sgemm_slice(const float* As, const float* Bs, int tx, int ty,
                                            uint64_t (&acc2)[8][Cfg::TN / 2]) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, TN = Cfg::TN;
    float4 fa[2][2], fb[2][Cfg::kChunks];
    auto load = [&](int k, int s) {
        fa[s][0] = *reinterpret_cast<const float4*>(As + k * Cfg::kAStride + ty * 4);
        fa[s][1] = *reinterpret_cast<const float4*>(As + k * Cfg::kAStride + BM / 2 + ty * 4);
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c)
            fb[s][c] = *reinterpret_cast<const float4*>(Bs + k * BN + Cfg::col(tx, c));
    };
    if constexpr (PF) load(0, 0);
#pragma unroll
    for (int k = 0; k < Cfg::BK; ++k) {
        const int s = PF ? (k & 1) : 0;
        if constexpr (PF) {
            if (k + 1 < Cfg::BK) load(k + 1, s ^ 1);
        } else {
            load(k, 0);
        }
        const float av[8] = {fa[s][0].x, fa[s][0].y, fa[s][0].z, fa[s][0].w,
                             fa[s][1].x, fa[s][1].y, fa[s][1].z, fa[s][1].w};
        uint64_t bp[TN / 2];
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
            bp[2 * c] = f32x2_pack(fb[s][c].x, fb[s][c].y);
            bp[2 * c + 1] = f32x2_pack(fb[s][c].z, fb[s][c].w);
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint64_t ai = f32x2_pack(av[i], av[i]);
#pragma unroll
            for (int p = 0; p < TN / 2; ++p) f32x2_fma(acc2[i][p], ai, bp[p]);
        }
    }
}

// acc (this thread's 8 x TN outputs) += A[m0.., kbeg..kend) x B[kbeg..kend, n0..).
// Two shared-memory buffers: the next slice is loaded into registers while
// the current one is multiplied, then stored to the other buffer, with one
// barrier per slice.  Ends with a barrier, so the caller may reuse shared
// memory.
template <class Cfg, bool EDGE, bool PF>
__device__ __forceinline__ void sgemm_mainloop(const SgArgs& a, int m0, int n0, int kbeg, int kend,
                                               float* smem, float (&acc)[8][Cfg::TN]) {
    constexpr int BK = Cfg::BK, TN = Cfg::TN;
    const int tx = threadIdx.x % Cfg::kTx;
    const int ty = threadIdx.x / Cfg::kTx;
    const int k_tiles = (kend - kbeg + BK - 1) / BK;
    const int k_full = (kend - kbeg) / BK;   // slices with no K tail

    // accumulators as column pairs (acc[i][2p], acc[i][2p+1])
    uint64_t acc2[8][TN / 2];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < TN / 2; ++p) acc2[i][p] = f32x2_pack(acc[i][2 * p], acc[i][2 * p + 1]);

    float* As0 = smem;
    float* Bs0 = smem + 2 * Cfg::kAFloats;
    float4 ra[Cfg::kAPer], rb[Cfg::kBPer];
    sgemm_load<Cfg, EDGE>(a, m0, n0, kbeg, kend, 0 >= k_full, ra, rb);
    sgemm_store_smem<Cfg>(As0, Bs0, ra, rb);
    __syncthreads();
    for (int kt = 0; kt < k_tiles; ++kt) {
        const float* As = As0 + (kt & 1) * Cfg::kAFloats;
        const float* Bs = Bs0 + (kt & 1) * Cfg::kBFloats;
        const bool more = kt + 1 < k_tiles;
        if (more)
            sgemm_load<Cfg, EDGE>(a, m0, n0, kbeg + (kt + 1) * BK, kend, kt + 1 >= k_full, ra, rb);
        sgemm_slice<Cfg, PF>(As, Bs, tx, ty, acc2);
        if (more)
            sgemm_store_smem<Cfg>(As0 + ((kt + 1) & 1) * Cfg::kAFloats, Bs0 + ((kt + 1) & 1) * Cfg::kBFloats,
                                  ra, rb);
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int p = 0; p < TN / 2; ++p) f32x2_unpack(acc2[i][p], acc[i][2 * p], acc[i][2 * p + 1]);
}

// This thread's outputs to C: row m0 + Cfg::row(ty, i), columns
// n0 + Cfg::col(tx, c) + 0..3, through the epilogue (alpha, beta, C type).
template <class Cfg, bool EDGE>
__device__ __forceinline__ void sgemm_store_c(const SgArgs& a, int m0, int n0,
                                              const float (&acc)[8][Cfg::TN]) {
    const int tx = threadIdx.x % Cfg::kTx;
    const int ty = threadIdx.x / Cfg::kTx;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int gm = m0 + Cfg::row(ty, i);
        if (EDGE && gm >= a.M) continue;
        const int64_t crow = static_cast<int64_t>(gm) * a.ldc;
#pragma unroll
        for (int c = 0; c < Cfg::kChunks; ++c) {
            const int gn = n0 + Cfg::col(tx, c);
            float v[4] = {acc[i][c * 4], acc[i][c * 4 + 1], acc[i][c * 4 + 2], acc[i][c * 4 + 3]};
            if (a.ab == 1) {
#pragma unroll
                for (int j = 0; j < 4; ++j) v[j] *= a.alpha;
            } else if (a.ab == 2) {
                // alpha * AB + beta * C, reading C only inside it
                if (!EDGE) {
                    const float4 cv = c_load4(a.C, crow + gn, a.ct);
                    v[0] = fmaf(a.alpha, v[0], a.beta * cv.x);
                    v[1] = fmaf(a.alpha, v[1], a.beta * cv.y);
                    v[2] = fmaf(a.alpha, v[2], a.beta * cv.z);
                    v[3] = fmaf(a.alpha, v[3], a.beta * cv.w);
                } else {
#pragma unroll
                    for (int j = 0; j < 4; ++j)
                        v[j] = fmaf(a.alpha, v[j],
                                    (gn + j < a.N) ? a.beta * c_load(a.C, crow + gn + j, a.ct) : 0.0f);
                }
            }
            if (!EDGE) {
                c_store4(a.C, crow + gn, v[0], v[1], v[2], v[3], a.ct);
            } else {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    if (gn + j < a.N) c_store(a.C, crow + gn + j, v[j], a.ct);
            }
        }
    }
}

// A piece of a cut tile: store this thread's partial outputs to workspace
// slot `slot` (its 2*TN float4, interleaved across threads so a warp's
// stores are contiguous) and count the arrival on the tile's counter; the
// piece that arrives last sums the tile's `nseg` slots first_slot.. in order
// (fixed order: the result does not depend on timing) and writes C.
template <class Cfg>
__device__ __forceinline__ void sgemm_piece(const SgArgs& a, int m0, int n0, bool edge,
                                            float (&acc)[8][Cfg::TN], int64_t slot, int64_t first_slot,
                                            int nseg, uint32_t* counter, uint32_t* s_last) {
    constexpr int TN = Cfg::TN;
    const int tid = threadIdx.x;
    constexpr int kQ = 2 * TN;          // float4 per thread (8 rows x TN columns)
    constexpr int kC = TN / 4;          // float4 per row
    constexpr int64_t kTile = Cfg::BM * Cfg::BN;
    float4* dst = reinterpret_cast<float4*>(a.ws + slot * kTile);
#pragma unroll
    for (int q = 0; q < kQ; ++q)
        dst[q * Cfg::kThreads + tid] = make_float4(acc[q / kC][(q % kC) * 4], acc[q / kC][(q % kC) * 4 + 1],
                                                   acc[q / kC][(q % kC) * 4 + 2], acc[q / kC][(q % kC) * 4 + 3]);
    __threadfence();
    __syncthreads();
    if (tid == 0) {
        const uint32_t old = atomicAdd(counter, 1u);
        *s_last = (old == static_cast<uint32_t>(nseg - 1)) ? 1u : 0u;
        if (*s_last) atomicExch(counter, 0u);   // ready for the next launch
    }
    __syncthreads();
    const bool last = *s_last != 0;
    __syncthreads();   // s_last may be reused by this CTA's next piece
    if (!last) return;
    __threadfence();
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < TN; ++j) acc[i][j] = 0.0f;
    for (int s2 = 0; s2 < nseg; ++s2) {
        const float4* src = reinterpret_cast<const float4*>(a.ws + (first_slot + s2) * kTile);
#pragma unroll
        for (int q = 0; q < kQ; ++q) {
            const float4 v = __ldcg(src + q * Cfg::kThreads + tid);
            acc[q / kC][(q % kC) * 4] += v.x;
            acc[q / kC][(q % kC) * 4 + 1] += v.y;
            acc[q / kC][(q % kC) * 4 + 2] += v.z;
            acc[q / kC][(q % kC) * 4 + 3] += v.w;
        }
    }
    if (!edge) sgemm_store_c<Cfg, false>(a, m0, n0, acc);
    else sgemm_store_c<Cfg, true>(a, m0, n0, acc);
}

// K steps [kb0, kb1) (of BK) of tile t: the product into acc (stream-K form).
template <class Cfg>
__device__ __forceinline__ void sgemm_tile_range(const SgArgs& a, int t, int kb0, int kb1, float* smem,
                                                 float (&acc)[8][Cfg::TN], int& m0, int& n0,
                                                 bool& edge) {
    m0 = (t / a.tiles_n) * Cfg::BM;
    n0 = (t - (t / a.tiles_n) * a.tiles_n) * Cfg::BN;
    const int kbeg = kb0 * Cfg::BK;
    const int kend = min(a.K, kb1 * Cfg::BK);
    edge = !(m0 + Cfg::BM <= a.M && n0 + Cfg::BN <= a.N);
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < Cfg::TN; ++j) acc[i][j] = 0.0f;
    if (!edge)
        sgemm_mainloop<Cfg, false, false>(a, m0, n0, kbeg, kend, smem, acc);
    else
        sgemm_mainloop<Cfg, true, false>(a, m0, n0, kbeg, kend, smem, acc);
}

// The CTA covering K step x of the stream-K range (CTA c owns
// [c*W/G, (c+1)*W/G)).
__device__ __forceinline__ int sg_owner(int64_t x, int64_t W, int G) {
    return static_cast<int>(((x + 1) * G - 1) / W);
}

// One stream-K segment of a CTA: K steps [kb0, kb1) of stream-K tile ts,
// which pieces first..last (CTA indices) share.
struct SgSeg {
    int ts, kb0, kb1, first, last;
};
constexpr int kSgMaxSegs = 4;   // a CTA's share is under two tiles' K steps: at most 3 segments

// Stream-K schedule: whole tiles cta, cta + G, ... below dp_tiles, then this
// CTA's contiguous share of the remaining tiles' K steps, cut at tile edges.
// The segments are listed in shared memory first, so that no schedule state
// stays live in registers across the main loop.
//
// This form is launched with programmatic stream serialization: the grid is
// exactly the CTAs that fit on the GPU at once, so a launch that starts while
// the previous kernel on the stream finishes only fills the slots that kernel
// leaves.  Listing the segments touches no global memory; every CTA waits
// for the previous kernel (griddepcontrol.wait) before its first load.
template <class Cfg>
__device__ __forceinline__ void sgemm_stream_k(const SgArgs& a, float* smem, uint32_t* s_last) {
    __shared__ SgSeg segs[kSgMaxSegs];
    __shared__ int nsegs;
    const int cta = blockIdx.x;
    grid_dep_launch_dependents();
    if (threadIdx.x == 0) {
        const int G = gridDim.x;
        const int64_t W = a.sk_iters, KB = a.kb_total;
        int64_t pos = static_cast<int64_t>(cta) * W / G;
        const int64_t end = static_cast<int64_t>(cta + 1) * W / G;
        int n = 0;
        while (pos < end && n < kSgMaxSegs) {
            const int64_t ts = pos / KB;                  // tile among the stream-K tiles
            const int64_t tile_end = (ts + 1) * KB;
            const int64_t stop = end < tile_end ? end : tile_end;
            SgSeg& sg = segs[n++];
            sg.ts = static_cast<int>(ts);
            sg.kb0 = static_cast<int>(pos - ts * KB);
            sg.kb1 = sg.kb0 + static_cast<int>(stop - pos);
            sg.first = sg_owner(ts * KB, W, G);
            sg.last = sg_owner(tile_end - 1, W, G);
            pos = stop;
        }
        nsegs = n;
    }
    grid_dep_wait();   // the previous kernel's writes (A or B may be its C) are visible
    float acc[8][Cfg::TN];
    int m0, n0;
    bool edge;
    for (int t = cta; t < a.dp_tiles; t += gridDim.x) {
        sgemm_tile_range<Cfg>(a, t, 0, a.kb_total, smem, acc, m0, n0, edge);
        if (!edge) sgemm_store_c<Cfg, false>(a, m0, n0, acc);
        else sgemm_store_c<Cfg, true>(a, m0, n0, acc);
    }
    __syncthreads();   // the segment list is written (the loop above may be empty)
    for (int i = 0; i < nsegs; ++i) {
        const SgSeg sg = segs[i];
        sgemm_tile_range<Cfg>(a, a.dp_tiles + sg.ts, sg.kb0, sg.kb1, smem, acc, m0, n0, edge);
        const SgSeg sd = segs[i];   // re-read after the main loop instead of keeping it live
        if (sd.first == sd.last) {
            if (!edge) sgemm_store_c<Cfg, false>(a, m0, n0, acc);
            else sgemm_store_c<Cfg, true>(a, m0, n0, acc);
        } else {
            const int64_t base = static_cast<int64_t>(sd.ts) * a.max_seg;
            sgemm_piece<Cfg>(a, m0, n0, edge, acc, base + (cta - sd.first), base, sd.last - sd.first + 1,
                             a.counters + sd.ts, s_last);
        }
    }
}

// One CTA per (tile, K slice).  With one slice the tile goes straight to C.
// With several, each slice stores its partial tile to the workspace and the
// CTA that finishes last sums the partials in slice order 0..S-1 (fixed
// order: the result does not depend on timing) and writes C.  The SK
// instantiation runs the persistent stream-K schedule instead (a separate
// kernel, so that its schedule costs the split kernel no registers).
// Shared memory (the operand buffers) is dynamic: Cfg::kSmemBytes.
template <class Cfg, bool SK>
__global__ void __launch_bounds__(Cfg::kThreads, Cfg::kMinBlocks) sgemm_kernel(const SgArgs a) {
    extern __shared__ __align__(16) float sg_smem[];
    __shared__ uint32_t s_last;
    if constexpr (SK) {
        sgemm_stream_k<Cfg>(a, sg_smem, &s_last);
        return;
    }
    const int u = blockIdx.x;
    const int tile = a.tile0 + u / a.splits;
    const int slice = u % a.splits;
    const int m0 = (tile / a.tiles_n) * Cfg::BM;
    const int n0 = (tile % a.tiles_n) * Cfg::BN;
    const int kbeg = slice * a.k_chunk;
    const int kend = min(a.K, kbeg + a.k_chunk);
    const bool edge = !(m0 + Cfg::BM <= a.M && n0 + Cfg::BN <= a.N);

    float acc[8][Cfg::TN];
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
        for (int j = 0; j < Cfg::TN; ++j) acc[i][j] = 0.0f;
    if (!edge)
        sgemm_mainloop<Cfg, false, true>(a, m0, n0, kbeg, kend, sg_smem, acc);
    else
        sgemm_mainloop<Cfg, true, true>(a, m0, n0, kbeg, kend, sg_smem, acc);

    if (a.splits == 1) {
        if (!edge) sgemm_store_c<Cfg, false>(a, m0, n0, acc);
        else sgemm_store_c<Cfg, true>(a, m0, n0, acc);
        return;
    }

    // partial tile of slice `slice`: slots of one tile are consecutive
    const int local_tile = u / a.splits;
    sgemm_piece<Cfg>(a, m0, n0, edge, acc, static_cast<int64_t>(u),
                     static_cast<int64_t>(local_tile) * a.splits, a.splits, a.counters + local_tile,
                     &s_last);
}

// Dynamic shared memory above 48 KB must be requested for the kernel (on
// the current device, before each launch: the setting belongs to a context).
template <class Cfg, bool SK>
static cudaError_t sgemm_prepare() {
    if (Cfg::kSmemBytes <= 48 * 1024) return cudaSuccess;
    return cudaFuncSetAttribute(sgemm_kernel<Cfg, SK>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg::kSmemBytes);
}

template <class Cfg>
static cudaError_t sgemm_go(const SgemmLaunch& L, cudaStream_t stream) {
    for (int i = 0; i < L.nparts; ++i) {
        const SgemmPart& part = L.parts[i];
        SgArgs a;
        a.A = L.A;
        a.B = L.B;
        a.C = L.C;
        a.M = static_cast<int>(L.M);
        a.N = static_cast<int>(L.N);
        a.K = static_cast<int>(L.K);
        a.lda = L.lda;
        a.ldb = L.ldb;
        a.ldc = L.ldc;
        a.ct = L.ct;
        a.tiles_n = static_cast<int>(ceil_div(L.N, Cfg::BN));
        a.tile0 = part.tile0;
        a.splits = part.splits;
        a.k_chunk = part.k_chunk;
        a.ab = L.ab;
        a.alpha = L.alpha;
        a.beta = L.beta;
        a.ws = L.ws;
        a.counters = L.counters;
        a.sk_mode = part.sk_mode;
        a.dp_tiles = part.dp_tiles;
        a.kb_total = static_cast<int>(ceil_div(L.K, kSgemmBK));
        a.sk_iters = part.sk_kblocks;
        a.max_seg = part.max_seg;
        if (part.sk_mode) {
            cudaError_t e = sgemm_prepare<Cfg, true>();
            if (e != cudaSuccess) return e;
            // the persistent stream-K grid starts early beside the previous
            // kernel (programmatic dependent launch; see sgemm_stream_k)
            cudaLaunchConfig_t cfg = {};
            cfg.gridDim = dim3(static_cast<unsigned>(part.grid));
            cfg.blockDim = dim3(Cfg::kThreads);
            cfg.dynamicSmemBytes = Cfg::kSmemBytes;
            cfg.stream = stream;
            cudaLaunchAttribute attr[1];
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
            e = cudaLaunchKernelEx(&cfg, sgemm_kernel<Cfg, true>, a);
            if (e != cudaSuccess) return e;
        } else {
            cudaError_t e = sgemm_prepare<Cfg, false>();
            if (e != cudaSuccess) return e;
            sgemm_kernel<Cfg, false><<<static_cast<unsigned>(part.tiles) * part.splits, Cfg::kThreads,
                                       Cfg::kSmemBytes, stream>>>(a);
        }
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// ------------------------------------------------------------- generic --

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) { return x; }
template <>
__device__ __forceinline__ float to_f32<__half>(__half x) { return __half2float(x); }
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) { return __bfloat162float(x); }

// 64 x 64 tile per CTA of 256 threads, 4 x 4 outputs per thread, K steps of
// 16, every access guarded: any alignment, any leading dimension.
template <typename T>
__global__ void __launch_bounds__(256)
generic_gemm_kernel(const T* __restrict__ A, const T* __restrict__ B, void* __restrict__ C, int ct,
                    int M, int N, int K, int64_t lda, int64_t ldb, int64_t ldc, int ab, float alpha,
                    float beta, int trans_a, int trans_b) {
    __shared__ float As[16][64 + 1];
    __shared__ float Bs[16][64 + 1];
    const int tid = threadIdx.x;
    const int tx = tid % 16, ty = tid / 16;
    const int m0 = blockIdx.y * 64, n0 = blockIdx.x * 64;
    float acc[4][4] = {};
    for (int k0 = 0; k0 < K; k0 += 16) {
        for (int l = tid; l < 64 * 16; l += 256) {
            const int r = l / 16, c = l % 16;     // A: 64 rows x 16 k
            const int gm = m0 + r, gk = k0 + c;
            // element (gm, gk) of op(A): A[gm][gk], or A[gk][gm] when A is stored transposed
            As[c][r] = (gm < M && gk < K)
                ? to_f32(A[trans_a ? static_cast<int64_t>(gk) * lda + gm : static_cast<int64_t>(gm) * lda + gk])
                : 0.0f;
            const int kr = l / 64, nc = l % 64;   // B: 16 k x 64 cols
            const int bk = k0 + kr, bn = n0 + nc;
            Bs[kr][nc] = (bk < K && bn < N)
                ? to_f32(B[trans_b ? static_cast<int64_t>(bn) * ldb + bk : static_cast<int64_t>(bk) * ldb + bn])
                : 0.0f;
        }
        __syncthreads();
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            float a[4], b[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) a[i] = As[k][ty + 16 * i];
#pragma unroll
            for (int j = 0; j < 4; ++j) b[j] = Bs[k][tx + 16 * j];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int gm = m0 + ty + 16 * i;
        if (gm >= M) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int gn = n0 + tx + 16 * j;
            if (gn < N) {
                const int64_t idx = static_cast<int64_t>(gm) * ldc + gn;
                float v = acc[i][j];
                if (ab == 1) v *= alpha;
                else if (ab == 2) v = fmaf(alpha, v, beta * c_load(C, idx, ct));
                c_store(C, idx, v, ct);
            }
        }
    }
}

// C = scale * C, or C = 0 without reading C when scale == 0.
__global__ void fill_scale_kernel(void* C, int ct, int64_t M, int64_t N, int64_t ldc, float scale) {
    const int64_t total = M * N;
    for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
         i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t r = i / N, c = i - r * N;
        const int64_t idx = r * ldc + c;
        c_store(C, idx, (scale == 0.0f) ? 0.0f : scale * c_load(C, idx, ct), ct);
    }
}

// ---------------------------------------------------------------- host --

// The SGEMM configurations built: (tile, micro-tile width).
template <class F>
static cudaError_t sgemm_dispatch(int bm, int bn, int tn, F&& f) {
    if (bm == 128 && bn == 128 && tn == 16) return f(SgemmCfg<128, 128, kSgemmBK, 16>{});
    if (bm == 128 && bn == 128 && tn == 8) return f(SgemmCfg<128, 128, kSgemmBK, 8>{});
    if (bm == 128 && bn == 64 && tn == 8) return f(SgemmCfg<128, 64, kSgemmBK, 8>{});
    if (bm == 64 && bn == 64 && tn == 8) return f(SgemmCfg<64, 64, kSgemmBK, 8>{});
    return cudaErrorInvalidValue;
}

bool sgemm_tile_supported(int bm, int bn, int tn) {
    return sgemm_dispatch(bm, bn, tn, [](auto) { return cudaSuccess; }) == cudaSuccess;
}

cudaError_t sgemm_blocks_per_sm(int bm, int bn, int tn, bool stream_k, int* n) {
    return sgemm_dispatch(bm, bn, tn, [&](auto c) {
        using Cfg = decltype(c);
        if (stream_k) {
            cudaError_t e = sgemm_prepare<Cfg, true>();
            if (e != cudaSuccess) return e;
            return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, sgemm_kernel<Cfg, true>, Cfg::kThreads,
                                                                 Cfg::kSmemBytes);
        }
        cudaError_t e = sgemm_prepare<Cfg, false>();
        if (e != cudaSuccess) return e;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(n, sgemm_kernel<Cfg, false>, Cfg::kThreads,
                                                             Cfg::kSmemBytes);
    });
}

int sgemm_k_step() { return kSgemmBK; }

cudaError_t sgemm_launch(const SgemmLaunch& L, cudaStream_t stream) {
    return sgemm_dispatch(L.bm, L.bn, L.tn, [&](auto c) { return sgemm_go<decltype(c)>(L, stream); });
}

cudaError_t generic_launch(int dtype, const void* A, const void* B, void* C, int ct, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           int ab, float alpha, float beta, int trans_a, int trans_b,
                           cudaStream_t stream) {
    dim3 grid(static_cast<unsigned>(ceil_div(N, 64)), static_cast<unsigned>(ceil_div(M, 64)));
    const int m = static_cast<int>(M), n = static_cast<int>(N), k = static_cast<int>(K);
    switch (dtype) {
        case 0:
            generic_gemm_kernel<__half><<<grid, 256, 0, stream>>>(
                static_cast<const __half*>(A), static_cast<const __half*>(B), C, ct, m, n, k, lda, ldb, ldc,
                ab, alpha, beta, trans_a, trans_b);
            break;
        case 1:
            generic_gemm_kernel<__nv_bfloat16><<<grid, 256, 0, stream>>>(
                static_cast<const __nv_bfloat16*>(A), static_cast<const __nv_bfloat16*>(B), C, ct, m, n,
                k, lda, ldb, ldc, ab, alpha, beta, trans_a, trans_b);
            break;
        default:
            generic_gemm_kernel<float><<<grid, 256, 0, stream>>>(
                static_cast<const float*>(A), static_cast<const float*>(B), C, ct, m, n, k, lda, ldb, ldc,
                ab, alpha, beta, trans_a, trans_b);
            break;
    }
    return cudaGetLastError();
}

cudaError_t fill_scale_launch(void* C, int ct, int64_t M, int64_t N, int64_t ldc, float scale,
                              cudaStream_t stream) {
    const int64_t total = M * N;
    int64_t blocks = ceil_div(total, 256);
    if (blocks > 4096) blocks = 4096;
    if (blocks < 1) blocks = 1;
    fill_scale_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(C, ct, M, N, ldc, scale);
    return cudaGetLastError();
}

}  // namespace gb300
