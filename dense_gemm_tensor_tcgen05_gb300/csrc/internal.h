// internal.h -- declarations shared by the library's translation units
// (host side only; not part of the public ABI).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace gb300 {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// One tensor-core GEMM launch, fully planned.
struct TcLaunch {
    const void* A;
    const void* B;
    void* C;            // element type ct
    int64_t M, N, K, lda, ldb, ldc;
    int ct;         // C's type: 0 = FP32, 1 = FP16, 2 = BF16
    int fmt;        // 0 = FP16, 1 = BF16, 2 = TF32 (FP32 storage), 3 = E4M3, 4 = E5M2
    int bn;         // tile width along the MMA N side
    int swap;       // 1: MMA M side runs along N of C (C^T = B^T A^T)
    int pair;       // 1: CTA-pair kernel (clusters of 2, 256 x bn tiles)
    int store_mode;    // 0: TMA stores when C allows them, 1: plain stores
    int ab;            // 0: C = AB; 1: C = alpha AB; 2: C = alpha AB + beta C
    float alpha, beta;
    int trans_a, trans_b;  // A stored K x M / B stored N x K (their transposes)
    int splits;     // K slices (split schedule)
    int sk_mode;    // 1: stream-K schedule (data-parallel tiles, then shared k-blocks)
    int dp_tiles;   // stream-K: tiles done whole
    int64_t sk_kblocks;  // stream-K: k-blocks shared out over the grid
    int sk_ctas;    // stream-K: CTAs (clusters) sharing them, 0 = the whole grid
    int max_seg;    // workspace slots per split tile
    int group;      // raster group height in tiles along the MMA M side
    int grid;       // CTAs (persistent); <= units
    float* ws;          // split-K partial tiles (splits * tiles * 128 * bn floats), or null
    uint32_t* counters; // split-K arrival counters (tiles * 4), zero between launches, or null
    // Self-test of the kernels' own bounded waits (gemm_ex_stall_selftest);
    // all zero for a normal launch.
    uint64_t wait_limit_ns;  // 0: the kernels' default limit
    int stall_cta;           // CTA (pair kernel: cluster) whose producer withholds one stage
    int stall_fill;          // 1 + index of the stage fill it withholds; 0: none
};

// Tile geometry helpers used by the planner and the launcher.
constexpr int kTcBM = 128;  // rows along the MMA M side (= tensor-memory lanes)
constexpr int kTcBK = 64;   // k per pipeline stage (64 16-bit elements = 128 bytes)
constexpr int kPairAtoms = 2;   // 128-byte K atoms per pipeline stage of the CTA-pair kernel

inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Stream-K schedule of the one-CTA kernel for `tiles` tiles of `kb_total`
// k-blocks on at most `sms` CTAs: fills dp_tiles, sk_kblocks, max_seg, grid
// of L and returns the number of tiles that need workspace slots.
int64_t tc_streamk_schedule(TcLaunch& L, int64_t tiles, int64_t kb_total, int sms);

// Tail-split schedule: whole waves of whole tiles, then each leftover tile
// cut into floor(sms / leftover) equal K pieces (one per CTA or cluster).
// Fills the same fields; returns the number of cut tiles (0: plain tiles).
int64_t tc_tailsplit_schedule(TcLaunch& L, int64_t tiles, int64_t kb_total, int sms);

// MMA kind of an input format (0: 16-bit, 1: TF32, 2: 8-bit), its element
// size in bytes, and the K elements one 128-byte stage row holds.
int tc_kind(int fmt);
int tc_elem_bytes(int fmt);
inline int tc_k_elems(int fmt) { return 128 / tc_elem_bytes(fmt); }

// Which (bn, swap, pair) kernels exist.
bool tc_config_supported(int bn, int swap, int pair);

// Most clusters of the CTA-pair kernel with tile width bn that can be resident
// at once on the current device.
cudaError_t tc_pair_max_clusters(int bn, int* n);

// Launch the tensor-core kernel.  Returns the first CUDA error (tensor-map
// encoding failures are reported as cudaErrorInvalidValue).
cudaError_t tc_gemm_launch(const TcLaunch& L, EncodeTiledFn encode, cudaStream_t stream);

// Launch the watchdog self-test kernel (a wait nothing satisfies, given up
// after limit_ns).
cudaError_t watchdog_selftest_launch(uint64_t limit_ns, cudaStream_t stream);

// Device address of this device's error word (cudaGetSymbolAddress on the
// tensor-core translation unit's __device__ variable).
cudaError_t tc_error_word(uint32_t** ptr);

// CUDA-core SGEMM: up to two launches over row-major linear tile ranges,
// each with its own K split (the second one spreads the last partial wave of
// tiles over more CTAs).
struct SgemmPart {
    int tile0;      // first linear tile
    int tiles;      // tiles in this launch
    int splits;     // K slices (split schedule)
    int sk_mode;    // 1: stream-K schedule (data-parallel tiles, then shared k-blocks)
    int dp_tiles;   // stream-K: tiles done whole
    int64_t sk_kblocks;  // stream-K: k-blocks shared out over the grid
    int max_seg;    // workspace slots per split tile per tile
    int k_chunk;    // K per slice (multiple of the kernel's K step)
    int grid;       // stream-K: CTAs (all resident at once)
};

struct SgemmLaunch {
    const float* A;
    const float* B;
    void* C;            // element type ct
    int64_t M, N, K, lda, ldb, ldc;
    int ct;             // C's type: 0 = FP32, 1 = FP16, 2 = BF16
    int bm, bn;
    int tn;             // columns of a thread's micro-tile: 8, or 16 (128 x 128 tiles of 128 threads)
    int nparts;
    SgemmPart parts[2];
    int ab;             // 0: C = AB; 1: C = alpha AB; 2: C = alpha AB + beta C
    float alpha, beta;
    float* ws;          // >= max over parts of tiles * splits * bm * bn floats (if any splits > 1)
    uint32_t* counters; // >= max over parts of tiles, zero between launches
};

bool sgemm_tile_supported(int bm, int bn, int tn);
// Resident CTAs per SM of the SGEMM kernel for a tile shape and micro-tile
// width (split or stream-K form).
cudaError_t sgemm_blocks_per_sm(int bm, int bn, int tn, bool stream_k, int* n);
int sgemm_k_step();
cudaError_t sgemm_launch(const SgemmLaunch& L, cudaStream_t stream);
cudaError_t generic_launch(int dtype, const void* A, const void* B, void* C, int ct, int64_t M,
                           int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                           int ab, float alpha, float beta, int trans_a, int trans_b,
                           cudaStream_t stream);
// C = beta * C (scale != 0) or C = 0 (scale == 0, C not read): the K == 0 result.
cudaError_t fill_scale_launch(void* C, int ct, int64_t M, int64_t N, int64_t ldc, float scale,
                              cudaStream_t stream);

}  // namespace gb300
