// tc_gemm.cu -- persistent, warp-specialised tensor-core GEMM for sm_103a.
//
// C = A x B (optionally alpha * A x B + beta * C) with FP16, BF16, TF32 or
// 8-bit floating-point A and B, FP32 accumulation, C stored as FP32, FP16 or
// BF16.  The tile decomposition is the one the pages describe for tensor
// cores -- loop over output tiles, accumulate the tile over K slices, store
// it once ("Tensor cores and matrix operations", "Complete Algorithm for
// Large Matrix Multiply") -- mapped onto Blackwell hardware:
//
//   * warp 0, one thread: TMA producer.  Per K step -- one 128-byte K atom
//     (64 16-bit, 32 TF32 or 128 8-bit elements), two in the CTA-pair
//     kernel -- it loads the rows of the MMA's A and B operands it needs,
//     128-byte swizzled, into a shared-memory ring; each stage has a "full"
//     mbarrier (TMA transaction bytes) and an "empty" mbarrier (released by
//     the MMA's commit).
//   * warp 1: allocates tensor memory (two BN-column FP32 accumulators of
//     128 lanes), and one thread issues tcgen05.mma (four per atom, each
//     32 bytes of K) and tcgen05.commit.
//   * warps 2-5: epilogue.  Each warp reads its 32 accumulator lanes with
//     tcgen05.ld and writes the results to C; the accumulator is double
//     buffered so the epilogue of one tile overlaps the next tile's main loop.
//
// Operand roles.  Without swap, the MMA's A operand is A (K contiguous:
// "K-major") and its B operand is B (N contiguous: "MN-major"), and
// tensor-memory lane = row of C.  With swap (small M) the kernel computes
// C^T = B^T A^T: the MMA's A operand is B (MN-major, 128 columns of C per
// tile) and its B operand is A (K-major, BN rows of C), and lane = column
// of C, so the epilogue's stores stay coalesced.
//
// Edges.  Loads never need a guard: TMA fills out-of-range elements of a box
// with zeros, so a K tail multiplies zeros and an M or N tail produces rows or
// columns that are never stored.  The epilogue decides once per 32-column
// chunk whether the chunk is whole (vector stores) or ragged (element-masked
// stores) -- a separate edge path instead of a guard in the inner loop, as
// "matmul_registers.cu" recommends for ragged shapes.
//
// Split-K.  A unit of work is (tile, K slice).  Each slice writes its FP32
// partial tile to a workspace and bumps a per-(tile, warp quarter) counter;
// the quarter that arrives last sums the partials in slice order 0..S-1 (a
// fixed order, so results do not depend on timing) and writes C.
//
// K order.  A CTA (or pair) walks K forwards in its even work items and
// backwards in its odd ones.  The work items of one wave run together, so
// the next wave's tiles start on the K slices of the operand panels that
// the previous wave read last, which are still in L2: at 8192^3 this cuts
// the DRAM reads of a launch by 18 %.  Only the order in which the K slices
// are loaded changes (the MMA thread still accumulates the stages in the
// order they arrive), so a given plan's results stay deterministic.
//
// Back-to-back launches.  Both kernels are launched with programmatic stream
// serialization: a launch may start while the previous kernel on the stream
// is still finishing.  It runs its prologue (barrier set-up, tensor-memory
// allocation, tensor-map prefetch) on the SMs that kernel has left, and the
// producer plans its first tile from the kernel parameters.  Only then does
// each role that touches global memory wait (griddepcontrol.wait) for the
// previous kernel to complete.  A stream of GEMMs then hides most of each
// launch's start-up; the order of every read and write of global memory is
// the same as with plain launches.
//
// Waits.  Every mbarrier wait gives up after kWaitLimitNs, sets a bit in the
// device error word and makes the whole CTA leave its loops; before exiting,
// the producer waits (bounded) for its own TMA copies and the MMA thread for
// its own MMAs, and tensor memory is freed on every path.  A self-test launch
// (TcArgs::stall_cta >= 0) shortens the limit and has one CTA's (or pair's)
// producer withhold the copies of one stage, so that this path runs: the
// MMA thread's wait for that stage runs out and the CTA aborts.

#include <algorithm>
#include <cstdio>
#include <cstring>

#include "cstore.cuh"
#include "internal.h"
#include "ptx.cuh"

namespace gb300 {

__device__ uint32_t g_tc_error;  // device error word; bits below

constexpr uint32_t kErrProducer = 1u, kErrMma = 2u, kErrEpilogue = 4u, kErrDrain = 8u,
                   kErrSelfTest = 16u;
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s: far above any legitimate wait
constexpr uint64_t kDrainLimitNs = 200000000ull;   // 0.2 s for copies already in flight
constexpr int kThreads = 192;
constexpr int kMmasPerStage = 4;   // MMAs per 128-byte K atom: each takes 32 bytes of K per row

// Elements of K per 128-byte stage row for an MMA kind (0: 16-bit, 1: TF32,
// 2: 8-bit).
__host__ __device__ constexpr int kind_k_elems(int kind) {
    return kind == 0 ? 64 : kind == 1 ? 32 : 128;
}
constexpr int kStoreStageBytes = 4 * 2 * 4096;   // epilogue staging: 4 warps x two 4 KiB buffers

struct TcArgs {
    void* C;                    // element type ct
    int64_t ldc;
    int32_t M, N;
    int32_t tiles_p, tiles_q;   // tiles along the MMA M side / N side
    int32_t num_units;          // tiles * splits (split schedule)
    int32_t splits, kb_total, kb_per_split;
    int32_t sk_mode;            // 1: data-parallel tiles, then stream-K over the rest
    int32_t dp_tiles;           // stream-K schedule: tiles done whole by one CTA each
    int64_t sk_kblocks;         // stream-K schedule: k-blocks shared out over the grid
    int32_t sk_ctas;            // CTAs (pair kernel: clusters) sharing them; 0 = the whole grid
    int32_t max_seg;            // workspace slots per split tile
    int32_t group;
    int32_t ct;                 // C's type: kCF32, kCF16 or kCBF16
    int32_t vec_store;          // C rows allow 4-element vector accesses (16 B FP32, 8 B 16-bit)
    int32_t tma_store;          // epilogue writes C through the TMA store map
    int32_t ab;                 // 0: C = AB; 1: alpha AB; 2: alpha AB + beta C
    float alpha, beta;
    int32_t p_kmajor;           // MMA A operand stored K-contiguous (else M/N-contiguous)
    int32_t q_kmajor;           // MMA B operand stored K-contiguous (else M/N-contiguous)
    uint32_t idesc;
    float* ws;
    uint32_t* counters;
    uint64_t wait_limit_ns;     // limit of every pipeline wait (kWaitLimitNs unless a self-test)
    int32_t stall_cta;          // self-test: this CTA (pair: cluster) withholds one stage; -1 none
    int32_t stall_fill;         // self-test: index of the stage fill it withholds
};

template <int BN, bool SWAP>
struct TcTraits {
    static constexpr int kPBytes = kTcBM * kTcBK * 2;   // MMA A operand per stage
    static constexpr int kQBytes = BN * kTcBK * 2;      // MMA B operand per stage
    static constexpr int kStageBytes = kPBytes + kQBytes;
    static constexpr int kStages = (BN == 256) ? 4 : (BN == 128) ? 6 : (BN == 64) ? 8
                                 : (BN == 32) ? 9 : 10;
    static constexpr int kTmemCols = (2 * BN < 32) ? 32 : 2 * BN;  // two accumulators
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kStoreBytes = SWAP ? 0 : kStoreStageBytes;   // epilogue staging
    static constexpr int kSmemBytes = 1024 /*alignment slack*/ + kStages * kStageBytes +
                                      kStoreBytes + kNumBars * 8 + 16;
    static_assert(BN % 16 == 0 && BN >= 16 && BN <= 256, "MMA N for M = 128");
    static_assert(SWAP ? (BN <= 64) : (BN >= 64 && BN % 64 == 0), "operand box shapes");
    static_assert((kTmemCols & (kTmemCols - 1)) == 0 && kTmemCols <= 512, "tensor memory");
    static_assert(kPBytes % 1024 == 0 && kQBytes % 1024 == 0, "1024-byte swizzle atoms");
    static_assert(kSmemBytes <= 227 * 1024, "shared memory per block");
    static_assert(kSmemBytes > 114 * 1024, "one CTA per SM keeps tensor memory uncontended");
};

struct WaitCtx {
    volatile uint32_t* abort_flag;
    uint64_t limit_ns;   // give up after this long
};

// Bounded wait: true when the phase of the given parity completed; false when
// the CTA is aborting (this wait gave up, or another role did).
__device__ __forceinline__ bool wait_phase(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                           uint32_t err_bit) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            *w.abort_flag = 1;
            atomicOr(&g_tc_error, err_bit);
            return false;
        }
    }
}

// Short bounded wait used only while draining before exit.
__device__ __forceinline__ void drain_wait(uint32_t bar, uint32_t parity) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > kDrainLimitNs) {
            atomicOr(&g_tc_error, kErrDrain);
            return;
        }
    }
}

// Tile -> (tile along MMA M side, tile along MMA N side).  Tiles are visited
// in groups of `group` tiles along the M side, column by column, so the CTAs
// working at one time share operand panels in L2.
__device__ __forceinline__ void tile_coords(const TcArgs& a, int tile, int& pb, int& qb) {
    const int group_tiles = a.group * a.tiles_q;
    const int g = tile / group_tiles;
    const int first_p = g * a.group;
    const int gsz = min(a.tiles_p - first_p, a.group);
    const int r = tile - g * group_tiles;
    pb = first_p + r % gsz;
    qb = r / gsz;
    // serpentine: odd groups sweep N backwards, so a group starts on the
    // operand panels the previous group used last (still in L2)
    if (g & 1) qb = a.tiles_q - 1 - qb;
}

// One piece of work for a CTA: k-blocks [kb0, kb1) of `tile`.  A tile cut
// into nseg > 1 pieces has its partial sums stored in workspace slot
// (slot, seg) and summed in seg order by whichever piece finishes last.
struct WorkItem {
    int tile, kb0, kb1, seg, nseg, slot;
};

// The CTA covering k-block x of the stream-K range (each CTA c owns
// [c*W/G, (c+1)*W/G)).
__device__ __forceinline__ int sk_owner(int64_t x, int64_t W, int G) {
    return static_cast<int>(((x + 1) * G - 1) / W);
}

// The sequence of work items of one CTA; the producer, the MMA thread and the
// epilogue each walk the same sequence.
//   split schedule: unit u = cta, cta + G, ... of tiles x splits equal slices;
//   stream-K schedule: whole tiles cta, cta + G, ... below dp_tiles, then a
//   contiguous share of the remaining tiles' k-blocks, cut at tile edges.
struct WorkIter {
    int cta, G;
    int next_u;
    int64_t pos, end;

    int Gs;   // CTAs (clusters) sharing the stream-K k-blocks: 0 .. Gs-1

    __device__ __forceinline__ WorkIter(const TcArgs& a, int cta_, int G_) : cta(cta_), G(G_), next_u(cta_) {
        Gs = a.sk_ctas > 0 ? a.sk_ctas : G;
        const bool shares = a.sk_kblocks > 0 && cta < Gs;
        pos = shares ? static_cast<int64_t>(cta) * a.sk_kblocks / Gs : 0;
        end = shares ? static_cast<int64_t>(cta + 1) * a.sk_kblocks / Gs : 0;
    }

    __device__ __forceinline__ bool next(const TcArgs& a, WorkItem& it) {
        if (!a.sk_mode) {
            if (next_u >= a.num_units) return false;
            const int u = next_u;
            next_u += G;
            it.tile = u / a.splits;
            it.seg = u - it.tile * a.splits;
            it.kb0 = it.seg * a.kb_per_split;
            it.kb1 = min(it.kb0 + a.kb_per_split, a.kb_total);
            it.nseg = a.splits;
            it.slot = it.tile;
            return true;
        }
        if (next_u < a.dp_tiles) {
            it.tile = next_u;
            next_u += G;
            it.kb0 = 0;
            it.kb1 = a.kb_total;
            it.seg = 0;
            it.nseg = 1;
            it.slot = 0;
            return true;
        }
        if (pos >= end) return false;
        const int64_t KB = a.kb_total;
        const int64_t ts = pos / KB;
        const int64_t tile_end = (ts + 1) * KB;
        const int64_t stop = end < tile_end ? end : tile_end;
        it.tile = a.dp_tiles + static_cast<int>(ts);
        it.kb0 = static_cast<int>(pos - ts * KB);
        it.kb1 = it.kb0 + static_cast<int>(stop - pos);
        const int first = sk_owner(ts * KB, a.sk_kblocks, Gs);
        const int last = sk_owner(tile_end - 1, a.sk_kblocks, Gs);
        it.seg = cta - first;
        it.nseg = last - first + 1;
        it.slot = static_cast<int>(ts);
        pos = stop;
        return true;
    }
};

// ---- split tiles ---------------------------------------------------------------
//
// A piece of a split tile is stored [column][row] (kTcBM rows a column), so
// a warp's loads and stores of one column are 32 consecutive floats.  The
// sum of a chunk of W columns over the n pieces is taken in piece order
// 0..n-1 (results do not depend on timing).  The loads of P pieces are
// issued before any is added, so a chunk costs one L2 round trip per P
// pieces instead of one per piece; callers pick P so that the P x W values
// fit in registers beside the rest of their epilogue.
template <int W, int P>
__device__ __forceinline__ void sum_pieces(float (&v)[W], const float* piece0, int n,
                                           int64_t piece_stride, int col0, int row) {
#pragma unroll
    for (int i = 0; i < W; ++i) v[i] = 0.0f;
    for (int s0 = 0; s0 < n; s0 += P) {
        float t[P][W];
#pragma unroll
        for (int j = 0; j < P; ++j) {
            if (s0 + j < n) {
                const float* src = piece0 + static_cast<int64_t>(s0 + j) * piece_stride;
#pragma unroll
                for (int i = 0; i < W; ++i) t[j][i] = __ldcg(src + (col0 + i) * kTcBM + row);
            }
        }
#pragma unroll
        for (int j = 0; j < P; ++j) {
            if (s0 + j < n) {
#pragma unroll
                for (int i = 0; i < W; ++i) v[i] += t[j][i];
            }
        }
    }
}

// ---- epilogue stores ----------------------------------------------------------

// W accumulator values of this thread's lane (`p` along the MMA M side),
// columns q0..q0+W-1 along the MMA N side.
template <bool SWAP, int W>
__device__ __forceinline__ void store_chunk(const TcArgs& a, const float (&v)[W], int p, int q0) {
    if (!SWAP) {
        // lane = row of C, chunk = W consecutive columns of that row.
        if (p >= a.M) return;
        const int64_t base = static_cast<int64_t>(p) * a.ldc + q0;
        if (a.vec_store && q0 + W <= a.N) {
#pragma unroll
            for (int i = 0; i < W; i += 4) c_store4(a.C, base + i, v[i], v[i + 1], v[i + 2], v[i + 3], a.ct);
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                if (q0 + i < a.N) c_store(a.C, base + i, v[i], a.ct);
        }
    } else {
        // lane = column of C, chunk = W consecutive rows; lanes of a warp
        // write 32 consecutive elements of each row.
        if (p >= a.N) return;
        const int64_t base = static_cast<int64_t>(q0) * a.ldc + p;
        if (q0 + W <= a.M) {
#pragma unroll
            for (int i = 0; i < W; ++i) c_store(a.C, base + static_cast<int64_t>(i) * a.ldc, v[i], a.ct);
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                if (q0 + i < a.M) c_store(a.C, base + static_cast<int64_t>(i) * a.ldc, v[i], a.ct);
        }
    }
}

// alpha * v + beta * C for W accumulator values of this thread (same
// coordinates as store_chunk), before they are stored.  C is read only when
// beta is in play (ab == 2), and only inside C.
template <bool SWAP, int W>
__device__ __forceinline__ void apply_ab(const TcArgs& a, float (&v)[W], int p, int q0) {
    if (!a.ab) return;
    const float alpha = a.alpha, beta = a.beta;
    if (a.ab == 1) {
#pragma unroll
        for (int i = 0; i < W; ++i) v[i] *= alpha;
        return;
    }
    if (!SWAP) {
        if (p >= a.M) return;   // never stored
        const int64_t base = static_cast<int64_t>(p) * a.ldc + q0;
        if (a.vec_store && q0 + W <= a.N) {
#pragma unroll
            for (int i = 0; i < W; i += 4) {
                const float4 c = c_load4(a.C, base + i, a.ct);
                v[i] = fmaf(alpha, v[i], beta * c.x);
                v[i + 1] = fmaf(alpha, v[i + 1], beta * c.y);
                v[i + 2] = fmaf(alpha, v[i + 2], beta * c.z);
                v[i + 3] = fmaf(alpha, v[i + 3], beta * c.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < W; ++i)
                v[i] = fmaf(alpha, v[i], (q0 + i < a.N) ? beta * c_load(a.C, base + i, a.ct) : 0.0f);
        }
    } else {
        if (p >= a.N) return;
        const int64_t base = static_cast<int64_t>(q0) * a.ldc + p;
#pragma unroll
        for (int i = 0; i < W; ++i)
            v[i] = fmaf(alpha, v[i],
                        (q0 + i < a.M) ? beta * c_load(a.C, base + static_cast<int64_t>(i) * a.ldc, a.ct) : 0.0f);
    }
}

// ---- operand layouts ----------------------------------------------------------
//
// Each MMA operand slice of R rows x 64 k sits in shared memory as R rows of
// 128 bytes either way:
//   K-major (K contiguous in memory): one TMA box {64 k, R rows} of a map
//     whose inner dimension is K;
//   MN-major (rows contiguous in memory): R/64 boxes {64 rows, 64 k} of a
//     map whose inner dimension is the row dimension, 8 KiB apart.
template <int R>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             bool kmajor, int r0, int k0) {
    if (kmajor) {
        tma_load_2d(dst, map, bar, k0, r0);
    } else {
#pragma unroll
        for (int j = 0; j < R / 64; ++j) tma_load_2d(dst + j * 8192, map, bar, r0 + 64 * j, k0);
    }
}

template <int R>
__device__ __forceinline__ void load_operand_pair(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar, bool kmajor, int r0, int k0) {
    if (kmajor) {
        tma_load_2d_pair(dst, map, bar, k0, r0);
    } else {
#pragma unroll
        for (int j = 0; j < R / 64; ++j) tma_load_2d_pair(dst + j * 8192, map, bar, r0 + 64 * j, k0);
    }
}

// Descriptor of k-step kk (16 k) of an operand slice: K-major steps 32 bytes
// along each 128-byte row; MN-major steps 16 rows of 128 bytes and finds the
// next 64-row block 8 KiB further (LBO).
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, bool kmajor, int kk) {
    return kmajor ? smem_desc_sw128(base + kk * 32, 16, 1024)
                  : smem_desc_sw128(base + kk * 2048, 8192, 1024);
}

// The MMA issuer's descriptors, kept in registers: the descriptor of stage s,
// k-step kk is the stage-0 descriptor plus (s * stage bytes) >> 4 plus
// kk * step in the start-address field (bits 0-13, address >> 4).  Shared
// memory addresses stay below 256 KiB, so the sum never carries out of the
// field, and the issue loop does no descriptor packing and no parameter loads.
struct DescIter {
    uint64_t base;   // descriptor of stage 0, k-step 0
    uint32_t step;   // one k-step in 16-byte units: 32 B (K-major) or 2 KiB (MN-major)
};

__device__ __forceinline__ DescIter desc_iter(uint32_t base, bool kmajor) {
    return DescIter{operand_desc(base, kmajor, 0), kmajor ? 2u : 128u};
}

// ---- TMA-store epilogue ------------------------------------------------------
//
// A warp's 32 accumulator rows x 32 columns (one chunk) go through a 4 KiB
// staging buffer in shared memory, written in the 128-byte swizzled order the
// store map expects (16-byte piece j of row r at piece j ^ (r % 8), which
// also keeps the warp's shared stores free of bank conflicts), and leave with
// one tensor store.  The TMA unit clips the box to C's bounds, so ragged
// tiles need no masks.  Each epilogue warp owns two buffers and alternates.

struct StoreStage {
    uint32_t base;   // this warp's two buffers, 1024-byte aligned
    int next;
};

__device__ __forceinline__ void stage_and_store32(StoreStage& st, const CUtensorMap* map_c,
                                                  const float (&v)[32], int lane, int col0, int row0,
                                                  int M, int N) {
    const uint32_t buf = st.base + static_cast<uint32_t>(st.next) * 4096u;
    if (lane == 0) bulk_wait_group_read<1>();   // the store issued from this buffer has read it
    __syncwarp();
    const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int j = 0; j < 8; ++j)
        st_shared_v4(rowaddr + (static_cast<uint32_t>(j ^ (lane & 7)) << 4), v[4 * j], v[4 * j + 1],
                     v[4 * j + 2], v[4 * j + 3]);
    fence_proxy_async_smem();
    __syncwarp();
    // A box wholly past C's end is skipped, and then the same buffer is used
    // again next time: only buffers that a store was issued from alternate, so
    // "at most one group still reading" always means the other buffer.
    if (row0 < M && col0 < N) {
        if (lane == 0) {
            tma_store_2d(map_c, buf, col0, row0);
            bulk_commit_group();
        }
        st.next ^= 1;
    }
}

// 16-bit C: a box is 32 rows x 64 columns (128 bytes a row, the same 4 KiB
// buffer), filled by two consecutive 32-column chunks -- the even chunk
// (col0 / 32 even) the row's first 64 bytes, the odd chunk the rest -- and
// stored after the odd one.  Tile widths are multiples of 64, so chunks come
// in such pairs.
__device__ __forceinline__ void stage_and_store16(StoreStage& st, const CUtensorMap* map_c,
                                                  const float (&v)[32], int lane, int col0, int row0,
                                                  int M, int N, int ct) {
    const uint32_t buf = st.base + static_cast<uint32_t>(st.next) * 4096u;
    const int half = (col0 >> 5) & 1;
    if (half == 0) {
        if (lane == 0) bulk_wait_group_read<1>();   // the store issued from this buffer has read it
        __syncwarp();
    }
    const uint32_t rowaddr = buf + static_cast<uint32_t>(lane) * 128u;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t piece = static_cast<uint32_t>(half * 4 + j);
        st_shared_v4_u32(rowaddr + ((piece ^ static_cast<uint32_t>(lane & 7)) << 4),
                         c_pack2(v[8 * j], v[8 * j + 1], ct), c_pack2(v[8 * j + 2], v[8 * j + 3], ct),
                         c_pack2(v[8 * j + 4], v[8 * j + 5], ct), c_pack2(v[8 * j + 6], v[8 * j + 7], ct));
    }
    if (half == 0) return;
    fence_proxy_async_smem();
    __syncwarp();
    const int box_col = col0 - 32;
    if (row0 < M && box_col < N) {
        if (lane == 0) {
            tma_store_2d(map_c, buf, box_col, row0);
            bulk_commit_group();
        }
        st.next ^= 1;
    }
}

__device__ __forceinline__ void stage_and_store(StoreStage& st, const CUtensorMap* map_c,
                                                const float (&v)[32], int lane, int col0, int row0,
                                                int M, int N, int ct) {
    if (ct == kCF32)
        stage_and_store32(st, map_c, v, lane, col0, row0, M, N);
    else
        stage_and_store16(st, map_c, v, lane, col0, row0, M, N, ct);
}

// ---- the kernel ---------------------------------------------------------------

template <int BN, bool SWAP, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_kernel(const __grid_constant__ CUtensorMap map_p, const __grid_constant__ CUtensorMap map_q,
               const __grid_constant__ CUtensorMap map_c, const TcArgs args) {
    using T = TcTraits<BN, SWAP>;
    constexpr int S = T::kStages;
    constexpr int CW = BN < 32 ? BN : 32;   // accumulator columns per tensor-memory load

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t store_base = smem_base + S * T::kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * T::kStageBytes + T::kStoreBytes);
    const uint32_t bar_base = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar_base + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar_base + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bar_base + 8u * (2 * S + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + T::kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 4);   // one arrival per epilogue warp
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_p);
        tma_prefetch_map(&map_q);
        if (!SWAP && args.tma_store) tma_prefetch_map(&map_c);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), T::kTmemCols);
        tmem_relinquish();
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touches only this CTA's shared and tensor memory and
    // the kernel parameters, so it may overlap the previous kernel on the
    // stream.  Each role that touches global memory waits for that kernel
    // (grid_dep_wait) before its first access: the producer before its first
    // copy, the epilogue warps before their first access to C or the
    // workspace.  The MMA thread touches none.
    grid_dep_launch_dependents();
    const WaitCtx wctx{abort_flag, args.wait_limit_ns};

    if (warp == 0) {
        // ------------------------------ TMA producer ------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;   // per-stage: armed at least once / parity
            bool ok = true;
            bool dep_ready = false;
            WorkIter wi(args, blockIdx.x, gridDim.x);
            WorkItem it;
            int items = 0;
            // self-test only: the fill index whose copies this CTA withholds
            const int stall = (static_cast<int>(blockIdx.x) == args.stall_cta) ? args.stall_fill : -1;
            int fills = 0;
            while (ok && wi.next(args, it)) {
                int pb, qb;
                tile_coords(args, it.tile, pb, qb);
                const int p0 = pb * kTcBM, q0 = qb * BN;
                // every other work item walks K backwards (see the kernel header)
                const bool k_down = (items++ & 1) != 0;
                for (int step = it.kb0; step < it.kb1; ++step) {
                    const int kb = k_down ? it.kb1 - 1 - (step - it.kb0) : step;
                    if (!wait_phase(empty_bar(stage), phase ^ 1u, wctx, kErrProducer)) {
                        ok = false;
                        break;
                    }
                    if (!dep_ready) {   // the first tile is planned; now the inputs may be read
                        grid_dep_wait();
                        dep_ready = true;
                    }
                    if (fills++ != stall) {
                        const uint32_t fb = full_bar(stage);
                        mbar_arrive_expect_tx(fb, T::kStageBytes);
                        armed |= 1u << stage;
                        armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        const uint32_t sp = smem_base + stage * T::kStageBytes;
                        const uint32_t sq = sp + T::kPBytes;
                        const int k0 = kb * kind_k_elems(KIND);
                        load_operand<kTcBM>(sp, &map_p, fb, args.p_kmajor, p0, k0);
                        load_operand<BN>(sq, &map_q, fb, args.q_kmajor, q0, k0);
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            // Every copy this thread issued has landed before the CTA exits.
            for (int s = 0; s < S; ++s)
                if (armed & (1u << s)) drain_wait(full_bar(s), (armed_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer --------------------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const DescIter dp = desc_iter(smem_base, args.p_kmajor);
            const DescIter dq = desc_iter(smem_base + T::kPBytes, args.q_kmajor);
            const uint32_t idesc = args.idesc;
            WorkIter wi(args, blockIdx.x, gridDim.x);
            WorkItem it;
            while (ok && wi.next(args, it)) {
                const int kb0 = it.kb0, kb1 = it.kb1;
                if (!wait_phase(acce_bar(acc), acc_phase ^ 1u, wctx, kErrMma)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(stage), phase, wctx, kErrMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t soff = static_cast<uint64_t>((stage * T::kStageBytes) >> 4);
#pragma unroll
                    for (int kk = 0; kk < kMmasPerStage; ++kk)
                        tc_mma<KIND>(d_tmem, dp.base + soff + kk * dp.step,
                                     dq.base + soff + kk * dq.step, idesc,
                                     (kb > kb0 || kk > 0) ? 1u : 0u);
                    tc_commit(empty_bar(stage));   // stage is free once these MMAs finish
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit(accf_bar(acc));          // accumulator ready for the epilogue
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            // Every MMA this thread issued has finished before tensor memory is freed.
            tc_commit(drain_bar);
            drain_wait(drain_bar, 0);
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue ----------------------------------
        grid_dep_wait();
        const int quarter = warp & 3;                 // tensor-memory lanes 32*quarter ..
        const int row = quarter * 32 + lane;          // lane within the 128-row tile
        StoreStage stg{store_base + static_cast<uint32_t>(warp - 2) * 8192u, 0};
        const bool tma_out = !SWAP && args.tma_store;
        int acc = 0;
        uint32_t acc_phase = 0;
        WorkIter wi(args, blockIdx.x, gridDim.x);
        WorkItem it;
        while (wi.next(args, it)) {
            int pb, qb;
            tile_coords(args, it.tile, pb, qb);
            bool ok = wait_phase(accf_bar(acc), acc_phase, wctx, kErrEpilogue);
            if (!__all_sync(0xffffffffu, ok)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after_sync();
            const uint32_t t_lane = tmem_base + static_cast<uint32_t>(acc * BN) +
                                    (static_cast<uint32_t>(quarter * 32) << 16);
            const int p = pb * kTcBM + row;
            const int q0 = qb * BN;
            const bool partial = it.nseg > 1;
            float* slot = partial
                ? args.ws + (static_cast<int64_t>(it.slot) * args.max_seg + it.seg) * (kTcBM * BN)
                : nullptr;
#pragma unroll 1
            for (int c = 0; c < BN / CW; ++c) {
                uint32_t r[CW];
                tmem_ld_lane_cols<CW>(t_lane + c * CW, r);
                tmem_wait_ld();
                if (c == BN / CW - 1) {
                    // accumulator fully read: hand it back to the MMA warp
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acce_bar(acc));
                }
                float v[CW];
#pragma unroll
                for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
                if (!partial) {
                    apply_ab<SWAP, CW>(args, v, p, q0 + c * CW);
                    if constexpr (!SWAP) {
                        if (tma_out) {
                            stage_and_store(stg, &map_c, v, lane, q0 + c * CW,
                                            pb * kTcBM + quarter * 32, args.M, args.N, args.ct);
                            continue;
                        }
                    }
                    store_chunk<SWAP, CW>(args, v, p, q0 + c * CW);
                } else {
                    // partial tile, laid out [column][row] so a warp's stores are
                    // 32 consecutive floats
#pragma unroll
                    for (int i = 0; i < CW; ++i) slot[(c * CW + i) * kTcBM + row] = v[i];
                }
            }
            if (partial) {
                __threadfence();
                __syncwarp();
                uint32_t last = 0;
                if (lane == 0) {
                    uint32_t* cnt = args.counters + it.slot * 4 + quarter;
                    last = (atomicAdd(cnt, 1u) == static_cast<uint32_t>(it.nseg - 1)) ? 1u : 0u;
                    if (last) atomicExch(cnt, 0u);   // ready for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    const float* base = args.ws + static_cast<int64_t>(it.slot) * args.max_seg * (kTcBM * BN);
#pragma unroll 1
                    for (int c = 0; c < BN / CW; ++c) {
                        float v[CW];
                        // the swapped epilogue needs more registers: fewer pieces in flight
                        sum_pieces<CW, SWAP ? (CW <= 16 ? 4 : 1) : 2>(v, base, it.nseg, kTcBM * BN, c * CW,
                                                                   row);
                        apply_ab<SWAP, CW>(args, v, p, q0 + c * CW);
                        if constexpr (!SWAP) {
                            if (tma_out) {
                                stage_and_store(stg, &map_c, v, lane, q0 + c * CW,
                                                pb * kTcBM + quarter * 32, args.M, args.N, args.ct);
                                continue;
                            }
                        }
                        store_chunk<SWAP, CW>(args, v, p, q0 + c * CW);
                    }
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (tma_out && lane == 0) bulk_wait_group<0>();   // every tensor store has completed
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, T::kTmemCols);
    }
}

// ---- the CTA-pair kernel ---------------------------------------------------------
//
// Same roles, pipeline and epilogue as tc_gemm_kernel, for a cluster of two
// CTAs that share one 256 x BN output tile.  Each CTA loads its own 128 rows
// of A and its own BN/2 columns of B per stage (so each SM moves two thirds
// of the bytes a 128 x BN tile needs), and the even CTA issues
// tcgen05.mma.cta_group::2 (M = 256), which reads both CTAs' shared memory
// and leaves each CTA's 128 rows of D in that CTA's tensor memory.
//   * both CTAs' TMA copies complete on the even CTA's "full" barrier, which
//     the even CTA arms for the bytes of both;
//   * the MMA commits are multicast to both CTAs' "empty", "acc_full" and
//     drain barriers;
//   * both CTAs' epilogue warps arrive on the even CTA's "acc_empty" (8
//     arrivals);
//   * a CTA that gives up a wait also raises the peer's abort flag, and a
//     cluster barrier keeps either CTA from freeing tensor memory or exiting
//     while the pair's MMAs may still read its shared memory.

constexpr uint64_t kPairDrainLimitNs = 3 * kWaitLimitNs;

// A stage holds kAtoms 128-byte swizzle atoms along K (each laid out exactly
// like a one-atom stage, kAtomBytes apart), so the MMA thread issues
// 4 * kAtoms MMAs per barrier wait and commit.  One thread issuing
// tcgen05.mma spends tens of cycles per instruction; with one atom per stage
// the wait, commit and loop overhead of each stage added up to more than the
// 512 tensor-core cycles the stage's four MMAs take, and the pipe ran dry.
template <int BN>
struct PairTraits {
    static constexpr int kAtoms = kPairAtoms;
    static constexpr int kAAtomBytes = kTcBM * 128;           // own 128 rows of A, one atom
    static constexpr int kBAtomBytes = (BN / 2) * 128;        // own BN/2 columns of B, one atom
    static constexpr int kABytes = kAtoms * kAAtomBytes;
    static constexpr int kBBytes = kAtoms * kBAtomBytes;
    static constexpr int kStageBytes = kABytes + kBBytes;
    static constexpr int kStoreBytes = kStoreStageBytes;
    // as many stages as fit beside the store buffers: 3 for BN 256, 4 for BN 128
    static constexpr int kStages = (227 * 1024 - 2048 - kStoreBytes) / kStageBytes;
    static constexpr int kTmemCols = 2 * BN;
    static constexpr int kNumBars = 2 * kStages + 5;
    static constexpr int kSmemBytes = 1024 + kStages * kStageBytes + kStoreBytes + kNumBars * 8 + 16;
    static_assert(BN == 256 || BN == 128, "pair tile widths");
    static_assert(kStages >= 3, "pipeline depth");
    static_assert(kSmemBytes <= 227 * 1024 && kSmemBytes > 114 * 1024, "shared memory");
    static_assert(kTmemCols <= 512, "tensor memory");
};

struct PairWaitCtx {
    volatile uint32_t* abort_flag;   // this CTA's flag (the peer may set it remotely)
    uint32_t peer_abort;             // shared::cluster address of the peer's flag
    uint64_t limit_ns;               // give up after this long
};

__device__ __forceinline__ void pair_raise_abort(const PairWaitCtx& w) {
    *w.abort_flag = 1;
    st_shared_cluster_u32(w.peer_abort, 1);
}

template <bool CLUSTER_SCOPE>
__device__ __forceinline__ bool pair_wait_phase(uint32_t bar, uint32_t parity,
                                                const PairWaitCtx& w, uint32_t err_bit) {
    auto test = [&]() {
        return CLUSTER_SCOPE ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
    };
    if (test()) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        if (test()) return true;
        if (*w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            atomicOr(&g_tc_error, err_bit);
            pair_raise_abort(w);
            return false;
        }
    }
}

template <int BN, int KIND>
__global__ void __launch_bounds__(kThreads, 1)
tc_gemm_pair_kernel(const __grid_constant__ CUtensorMap map_a, const __grid_constant__ CUtensorMap map_b,
                    const __grid_constant__ CUtensorMap map_c, const TcArgs args) {
    using T = PairTraits<BN>;
    constexpr int S = T::kStages;
    constexpr int CW = 32;

    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const uint32_t smem_base = smem_u32(smem);
    const uint32_t store_base = smem_base + S * T::kStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + S * T::kStageBytes + T::kStoreBytes);
    const uint32_t bar_base = smem_u32(bars);
    auto full_bar = [&](int s) { return bar_base + 8u * s; };
    auto empty_bar = [&](int s) { return bar_base + 8u * (S + s); };
    auto accf_bar = [&](int b) { return bar_base + 8u * (2 * S + b); };
    auto acce_bar = [&](int b) { return bar_base + 8u * (2 * S + 2 + b); };
    const uint32_t drain_bar = bar_base + 8u * (2 * S + 4);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + T::kNumBars);
    volatile uint32_t* abort_flag = tmem_slot + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(accf_bar(b), 1);
            mbar_init(acce_bar(b), 8);   // four epilogue warps in each CTA
        }
        mbar_init(drain_bar, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_map(&map_a);
        tma_prefetch_map(&map_b);
        if (args.tma_store) tma_prefetch_map(&map_c);
    }
    if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), T::kTmemCols);
        tmem_relinquish_pair();
    }
    tc_fence_before_sync();
    cluster_sync();   // both CTAs' barriers exist and tensor memory is allocated
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;
    // Everything above touches only this CTA's shared and tensor memory and
    // the kernel parameters, so it may overlap the previous kernel on the
    // stream.  Each role that touches global memory waits for that kernel
    // (grid_dep_wait) before its first access: the producer before its first
    // copy, the epilogue warps before their first access to C or the
    // workspace.  The MMA thread touches none.
    grid_dep_launch_dependents();
    const PairWaitCtx wctx{abort_flag,
                           mapa_shared(smem_u32(const_cast<uint32_t*>(abort_flag)), rank ^ 1u),
                           args.wait_limit_ns};
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(cluster_count_x());

    if (warp == 0) {
        // ------------------------------ TMA producer (both CTAs) ------------------
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            uint32_t armed = 0, armed_parity = 0;
            bool ok = true;
            bool dep_ready = false;
            WorkIter wi(args, cid, ncl);
            WorkItem it;
            int items = 0;
            // self-test only: both CTAs of the stalled pair withhold the same
            // fill (the even CTA does not arm it, the odd CTA copies nothing
            // into it), so no copy is left in flight for that stage
            const int stall = (cid == args.stall_cta) ? args.stall_fill : -1;
            int fills = 0;
            while (ok && wi.next(args, it)) {
                int pb, qb;
                tile_coords(args, it.tile, pb, qb);
                const int m0 = pb * (2 * kTcBM) + static_cast<int>(rank) * kTcBM;
                const int n0 = qb * BN + static_cast<int>(rank) * (BN / 2);
                // every other work item walks K backwards (see the kernel header)
                const bool k_down = (items++ & 1) != 0;
                for (int step = it.kb0; step < it.kb1; ++step) {
                    const int ks = k_down ? it.kb1 - 1 - (step - it.kb0) : step;
                    if (!pair_wait_phase<false>(empty_bar(stage), phase ^ 1u, wctx, kErrProducer)) {
                        ok = false;
                        break;
                    }
                    if (!dep_ready) {   // the first tile is planned; now the inputs may be read
                        grid_dep_wait();
                        dep_ready = true;
                    }
                    if (fills++ != stall) {
                        if (leader) {
                            // both CTAs' bytes complete on this barrier
                            mbar_arrive_expect_tx(full_bar(stage), 2 * T::kStageBytes);
                            armed |= 1u << stage;
                            armed_parity = (armed_parity & ~(1u << stage)) | (phase << stage);
                        }
                        const uint32_t fb = mapa_shared(full_bar(stage), 0);
                        const uint32_t sa = smem_base + stage * T::kStageBytes;
                        const uint32_t sb = sa + T::kABytes;
                        // atoms past K are fetched too: the copy fills them with zeros
#pragma unroll
                        for (int j = 0; j < T::kAtoms; ++j) {
                            const int k0 = (ks * T::kAtoms + j) * kind_k_elems(KIND);
                            load_operand_pair<kTcBM>(sa + j * T::kAAtomBytes, &map_a, fb,
                                                     args.p_kmajor, m0, k0);
                            load_operand_pair<BN / 2>(sb + j * T::kBAtomBytes, &map_b, fb,
                                                      args.q_kmajor, n0, k0);
                        }
                    }
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (leader)
                for (int s = 0; s < S; ++s)
                    if (armed & (1u << s)) drain_wait(full_bar(s), (armed_parity >> s) & 1u);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------ MMA issuer (even CTA) ---------------------
        if (lane == 0 && leader) {
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            const DescIter da = desc_iter(smem_base, args.p_kmajor);
            const DescIter db = desc_iter(smem_base + T::kABytes, args.q_kmajor);
            const uint32_t idesc = args.idesc;
            WorkIter wi(args, cid, ncl);
            WorkItem it;
            while (ok && wi.next(args, it)) {
                const int kb0 = it.kb0, kb1 = it.kb1;
                if (!pair_wait_phase<true>(acce_bar(acc), acc_phase ^ 1u, wctx, kErrMma)) break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int ks = kb0; ks < kb1; ++ks) {
                    if (!pair_wait_phase<false>(full_bar(stage), phase, wctx, kErrMma)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after_sync();
                    const uint64_t soff = static_cast<uint64_t>((stage * T::kStageBytes) >> 4);
#pragma unroll
                    for (int j = 0; j < T::kAtoms; ++j) {
                        const uint64_t ao = soff + ((j * T::kAAtomBytes) >> 4);
                        const uint64_t bo = soff + ((j * T::kBAtomBytes) >> 4);
#pragma unroll
                        for (int kk = 0; kk < kMmasPerStage; ++kk)
                            tc_mma_pair<KIND>(d_tmem, da.base + ao + kk * da.step,
                                              db.base + bo + kk * db.step, idesc,
                                              (ks > kb0 || j > 0 || kk > 0) ? 1u : 0u);
                    }
                    tc_commit_pair_multicast(empty_bar(stage), 0x3);
                    if (++stage == S) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (!ok) break;
                tc_commit_pair_multicast(accf_bar(acc), 0x3);
                acc ^= 1;
                if (acc == 0) acc_phase ^= 1u;
            }
            tc_commit_pair_multicast(drain_bar, 0x3);   // both CTAs learn when every MMA is done
        }
        __syncwarp();
    } else {
        // ------------------------------ epilogue (both CTAs) ----------------------
        grid_dep_wait();
        const int quarter = warp & 3;
        const int row = quarter * 32 + lane;
        StoreStage stg{store_base + static_cast<uint32_t>(warp - 2) * 8192u, 0};
        int acc = 0;
        uint32_t acc_phase = 0;
        WorkIter wi(args, cid, ncl);
        WorkItem it;
        while (wi.next(args, it)) {
            int pb, qb;
            tile_coords(args, it.tile, pb, qb);
            bool ok = pair_wait_phase<false>(accf_bar(acc), acc_phase, wctx, kErrEpilogue);
            if (!__all_sync(0xffffffffu, ok)) {
                if (lane == 0) pair_raise_abort(wctx);
                break;
            }
            tc_fence_after_sync();
            const uint32_t t_lane = tmem_base + static_cast<uint32_t>(acc * BN) +
                                    (static_cast<uint32_t>(quarter * 32) << 16);
            const int row0 = pb * (2 * kTcBM) + static_cast<int>(rank) * kTcBM;   // this CTA's rows
            const int p = row0 + row;
            const int q0 = qb * BN;
            // A piece of a stream-K tile: each CTA owns its 128 rows of the
            // workspace slot (tile, piece), laid out [column][row].
            const bool partial = it.nseg > 1;
            float* slot = partial
                ? args.ws + ((static_cast<int64_t>(it.slot) * args.max_seg + it.seg) * 2 + rank) *
                                (kTcBM * BN)
                : nullptr;
#pragma unroll 1
            for (int c = 0; c < BN / CW; ++c) {
                uint32_t r[CW];
                tmem_ld_lane_cols<CW>(t_lane + c * CW, r);
                tmem_wait_ld();
                if (c == BN / CW - 1) {
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive_cluster(mapa_shared(acce_bar(acc), 0));
                }
                float v[CW];
#pragma unroll
                for (int i = 0; i < CW; ++i) v[i] = __uint_as_float(r[i]);
                if (partial) {
#pragma unroll
                    for (int i = 0; i < CW; ++i) slot[(c * CW + i) * kTcBM + row] = v[i];
                    continue;
                }
                apply_ab<false, CW>(args, v, p, q0 + c * CW);
                if (args.tma_store)
                    stage_and_store(stg, &map_c, v, lane, q0 + c * CW, row0 + quarter * 32, args.M,
                                    args.N, args.ct);
                else
                    store_chunk<false, CW>(args, v, p, q0 + c * CW);
            }
            if (partial) {
                // the last piece to arrive (per CTA and warp quarter) sums the
                // pieces in piece order, so results do not depend on timing
                __threadfence();
                __syncwarp();
                uint32_t last = 0;
                if (lane == 0) {
                    uint32_t* cnt = args.counters + it.slot * 8 + rank * 4 + quarter;
                    last = (atomicAdd(cnt, 1u) == static_cast<uint32_t>(it.nseg - 1)) ? 1u : 0u;
                    if (last) atomicExch(cnt, 0u);   // ready for the next launch
                }
                last = __shfl_sync(0xffffffffu, last, 0);
                if (last) {
                    __threadfence();
                    // pieces of this CTA's rows: slot (tile, piece, CTA), pieces 2 slots apart
                    const float* base =
                        args.ws + (static_cast<int64_t>(it.slot) * args.max_seg * 2 + rank) * (kTcBM * BN);
#pragma unroll 1
                    for (int c = 0; c < BN / CW; ++c) {
                        float v[CW];
                        sum_pieces<CW, 2>(v, base, it.nseg, 2 * kTcBM * BN, c * CW, row);
                        apply_ab<false, CW>(args, v, p, q0 + c * CW);
                        if (args.tma_store)
                            stage_and_store(stg, &map_c, v, lane, q0 + c * CW, row0 + quarter * 32,
                                            args.M, args.N, args.ct);
                        else
                            store_chunk<false, CW>(args, v, p, q0 + c * CW);
                    }
                }
            }
            acc ^= 1;
            if (acc == 0) acc_phase ^= 1u;
        }
        if (args.tma_store && lane == 0) bulk_wait_group<0>();
        __syncwarp();
    }

    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1 && lane == 0) {
        // the even CTA's last commit: every pair MMA (which may read this CTA's
        // shared memory and write its tensor memory) has finished
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(drain_bar, 0)) {
            if (globaltimer_ns() - t0 > kPairDrainLimitNs) {
                atomicOr(&g_tc_error, kErrDrain);
                break;
            }
        }
        if (*abort_flag) {
            // give copies issued just before an abort time to land
            const uint64_t t1 = globaltimer_ns();
            while (globaltimer_ns() - t1 < 50000ull) {
            }
        }
    }
    __syncwarp();
    tc_fence_before_sync();
    cluster_sync();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc_pair(tmem_base, T::kTmemCols);
    }
}

// ---- watchdog self-test --------------------------------------------------------
//
// One thread waits, through the same bounded wait the GEMM kernels use, on an
// mbarrier that nothing ever arrives on.  The wait gives up after limit_ns,
// records kErrSelfTest in the device error word and the kernel returns: the
// host sees GEMM_ERR_DEVICE_TIMEOUT from gemm_device_error() and the context
// stays usable.

__global__ void watchdog_selftest_kernel(uint64_t limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_barrier_init();
        const WaitCtx w{&abort_flag, limit_ns};
        wait_phase(smem_u32(&bar), 0, w, kErrSelfTest);
    }
}

cudaError_t watchdog_selftest_launch(uint64_t limit_ns, cudaStream_t stream) {
    watchdog_selftest_kernel<<<1, 32, 0, stream>>>(limit_ns);
    return cudaGetLastError();
}

// ---- host side --------------------------------------------------------------------

int64_t tc_streamk_schedule(TcLaunch& L, int64_t tiles, int64_t kb_total, int sms) {
    int64_t G = sms;
    int64_t dp = 0;
    if (tiles >= G) dp = (tiles % G == 0) ? tiles : (tiles / G - 1) * G;
    int64_t W = (tiles - dp) * kb_total;
    if (W > 0 && W < G) G = W;            // every CTA gets at least one k-block
    if (dp > 0 && W == 0) G = std::min<int64_t>(G, tiles);
    L.sk_mode = 1;
    L.dp_tiles = static_cast<int>(dp);
    L.sk_kblocks = W;
    L.grid = static_cast<int>(std::max<int64_t>(G, 1));
    int max_seg = 1;
    const int64_t sk_tiles = tiles - dp;
    for (int64_t ts = 0; ts < sk_tiles; ++ts) {
        const int64_t first = ((ts * kb_total + 1) * G - 1) / W;
        const int64_t last = (((ts + 1) * kb_total) * G - 1) / W;
        max_seg = std::max<int>(max_seg, static_cast<int>(last - first + 1));
    }
    L.max_seg = max_seg;
    L.splits = 1;
    return max_seg > 1 ? sk_tiles : 0;
}

int64_t tc_tailsplit_schedule(TcLaunch& L, int64_t tiles, int64_t kb_total, int sms) {
    // whole waves of whole tiles; the tiles left over (fewer than a wave) are
    // each cut into S = floor(sms / left) equal K pieces, one per CTA, so the
    // last wave runs S times shorter on S times as many CTAs
    const int64_t G = sms;
    const int64_t dp = (tiles / G) * G;
    const int64_t left = tiles - dp;
    const int64_t S = left > 0 ? std::min<int64_t>(G / left, kb_total) : 0;
    L.splits = 1;
    L.max_seg = 1;
    L.sk_ctas = 0;
    if (left == 0 || S < 2) {   // nothing to gain: plain whole tiles
        L.sk_mode = 0;
        L.dp_tiles = 0;
        L.sk_kblocks = 0;
        L.grid = static_cast<int>(std::min<int64_t>(tiles, G));
        return 0;
    }
    const int64_t W = left * kb_total;
    const int64_t Gs = left * S;
    L.sk_mode = 1;
    L.dp_tiles = static_cast<int>(dp);
    L.sk_kblocks = W;
    L.sk_ctas = static_cast<int>(Gs);
    L.grid = static_cast<int>(G);
    int max_seg = 1;
    for (int64_t ts = 0; ts < left; ++ts) {
        const int64_t first = ((ts * kb_total + 1) * Gs - 1) / W;
        const int64_t last = (((ts + 1) * kb_total) * Gs - 1) / W;
        max_seg = std::max<int>(max_seg, static_cast<int>(last - first + 1));
    }
    L.max_seg = max_seg;
    return left;
}

bool tc_config_supported(int bn, int swap, int pair) {
    if (pair) return !swap && (bn == 128 || bn == 256);
    if (swap) return bn == 16 || bn == 32 || bn == 64;
    return bn == 64 || bn == 128 || bn == 256;
}

template <int BN>
static cudaLaunchConfig_t pair_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = PairTraits<BN>::kSmemBytes;
    cfg.stream = stream;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cfg;
}

template <int BN>
static cudaError_t pair_max_clusters_for(int* n) {
    auto kern = tc_gemm_pair_kernel<BN, 0>;   // residency is the same for every kind
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairTraits<BN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<BN>(2, nullptr, attr);
    return cudaOccupancyMaxActiveClusters(n, kern, &cfg);
}

cudaError_t tc_pair_max_clusters(int bn, int* n) {
    *n = 0;
    if (bn == 256) return pair_max_clusters_for<256>(n);
    if (bn == 128) return pair_max_clusters_for<128>(n);
    return cudaErrorInvalidValue;
}

cudaError_t tc_error_word(uint32_t** ptr) {
    return cudaGetSymbolAddress(reinterpret_cast<void**>(ptr), g_tc_error);
}

// fmt: 0 FP16, 1 BF16, 2 TF32 (FP32 storage), 3 E4M3, 4 E5M2.
int tc_kind(int fmt) { return fmt <= 1 ? 0 : fmt == 2 ? 1 : 2; }
int tc_elem_bytes(int fmt) { return fmt <= 1 ? 2 : fmt == 2 ? 4 : 1; }

static bool encode_map(EncodeTiledFn encode, CUtensorMap* map, int fmt, const void* base,
                       uint64_t inner, uint64_t outer, uint64_t ld_elems, uint32_t box_inner,
                       uint32_t box_outer) {
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {ld_elems * tc_elem_bytes(fmt)};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapDataType dt =
        fmt == 0 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
        : fmt == 1 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
        : fmt == 2 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    CUresult r = encode(map, dt, 2, const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int BN, bool SWAP, int KIND>
static cudaError_t launch_cfg(const TcLaunch& L, const CUtensorMap& mp, const CUtensorMap& mq,
                              const CUtensorMap& mc, const TcArgs& args, cudaStream_t stream) {
    using T = TcTraits<BN, SWAP>;
    auto kern = tc_gemm_kernel<BN, SWAP, KIND>;
    // The attribute is per device; setting it every call is cheap and keeps
    // multi-device use correct.
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(L.grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = T::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, mp, mq, mc, args);
}

template <int BN, int KIND>
static cudaError_t launch_pair(const TcLaunch& L, const CUtensorMap& ma, const CUtensorMap& mb,
                               const CUtensorMap& mc, const TcArgs& args, cudaStream_t stream) {
    auto kern = tc_gemm_pair_kernel<BN, KIND>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         PairTraits<BN>::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchAttribute attr[2];
    cudaLaunchConfig_t cfg = pair_config<BN>(L.grid, stream, attr);
    return cudaLaunchKernelEx(&cfg, kern, ma, mb, mc, args);
}

template <int KIND>
static cudaError_t dispatch_kind(const TcLaunch& L, const CUtensorMap& map_a, const CUtensorMap& map_b,
                                 const CUtensorMap& mp, const CUtensorMap& mq, const CUtensorMap& map_c,
                                 const TcArgs& a, cudaStream_t stream) {
    if (L.pair) {
        switch (L.bn) {
            case 128: return launch_pair<128, KIND>(L, map_a, map_b, map_c, a, stream);
            case 256: return launch_pair<256, KIND>(L, map_a, map_b, map_c, a, stream);
        }
        return cudaErrorInvalidValue;
    }
    if (!L.swap) {
        switch (L.bn) {
            case 64: return launch_cfg<64, false, KIND>(L, mp, mq, map_c, a, stream);
            case 128: return launch_cfg<128, false, KIND>(L, mp, mq, map_c, a, stream);
            case 256: return launch_cfg<256, false, KIND>(L, mp, mq, map_c, a, stream);
        }
    } else {
        switch (L.bn) {
            case 16: return launch_cfg<16, true, KIND>(L, mp, mq, map_c, a, stream);
            case 32: return launch_cfg<32, true, KIND>(L, mp, mq, map_c, a, stream);
            case 64: return launch_cfg<64, true, KIND>(L, mp, mq, map_c, a, stream);
        }
    }
    return cudaErrorInvalidValue;
}

cudaError_t tc_gemm_launch(const TcLaunch& L, EncodeTiledFn encode, cudaStream_t stream) {
    if (!tc_config_supported(L.bn, L.swap, L.pair)) return cudaErrorInvalidValue;
    if (L.pair && (L.splits != 1 || (L.grid & 1))) return cudaErrorInvalidValue;
    // Operand roles: the MMA's A operand (128 rows) is op(A) -- or op(B)^T with
    // swap -- and its B operand (BN rows; BN/2 per CTA in pairs) the other.
    // A stored plain (M x K, trans_a = 0) is K-major; stored transposed
    // (K x M) it is M-major.  B stored plain (K x N) is N-major; stored
    // transposed (N x K) it is K-major.
    const bool a_kmajor = !L.trans_a, b_kmajor = L.trans_b != 0;
    const uint32_t a_rows = L.swap ? static_cast<uint32_t>(L.bn) : kTcBM;
    const uint32_t b_rows = L.swap ? kTcBM : static_cast<uint32_t>(L.pair ? L.bn / 2 : L.bn);
    if ((!a_kmajor && a_rows % 64) || (!b_kmajor && b_rows % 64)) return cudaErrorInvalidValue;
    // TF32 and 8-bit operands are read K-major only
    if (tc_kind(L.fmt) != 0 && (!a_kmajor || !b_kmajor)) return cudaErrorInvalidValue;
    const uint32_t ke = static_cast<uint32_t>(kind_k_elems(tc_kind(L.fmt)));
    CUtensorMap map_a, map_b;
    const bool ok_a = a_kmajor ? encode_map(encode, &map_a, L.fmt, L.A, L.K, L.M, L.lda, ke, a_rows)
                               : encode_map(encode, &map_a, L.fmt, L.A, L.M, L.K, L.lda, 64, 64);
    const bool ok_b = b_kmajor ? encode_map(encode, &map_b, L.fmt, L.B, L.K, L.N, L.ldb, ke, b_rows)
                               : encode_map(encode, &map_b, L.fmt, L.B, L.N, L.K, L.ldb, 64, 64);
    if (!ok_a || !ok_b) return cudaErrorInvalidValue;

    TcArgs a;
    a.C = L.C;
    a.ldc = L.ldc;
    a.M = static_cast<int32_t>(L.M);
    a.N = static_cast<int32_t>(L.N);
    const int64_t pe = L.swap ? L.N : L.M;
    const int64_t qe = L.swap ? L.M : L.N;
    a.tiles_p = static_cast<int32_t>(ceil_div(pe, L.pair ? 2 * kTcBM : kTcBM));
    a.tiles_q = static_cast<int32_t>(ceil_div(qe, L.bn));
    // k-steps: one pipeline stage of K (one 128-byte atom; the pair kernel's
    // stages hold kPairAtoms)
    a.kb_total = static_cast<int32_t>(
        ceil_div(L.K, kind_k_elems(tc_kind(L.fmt)) * (L.pair ? kPairAtoms : 1)));
    a.splits = L.splits;
    a.kb_per_split = static_cast<int32_t>(ceil_div(a.kb_total, L.splits));
    a.num_units = a.tiles_p * a.tiles_q * L.splits;
    a.sk_mode = L.sk_mode;
    a.dp_tiles = L.dp_tiles;
    a.sk_kblocks = L.sk_kblocks;
    a.sk_ctas = L.sk_ctas;
    a.max_seg = L.sk_mode ? L.max_seg : L.splits;
    a.group = L.group;
    a.ct = L.ct;
    // 4-element vector accesses: 16 bytes of FP32 or 8 bytes of a 16-bit type
    const uintptr_t c_addr = reinterpret_cast<uintptr_t>(L.C);
    const uintptr_t vec_align = L.ct == kCF32 ? 15 : 7;
    a.vec_store = ((c_addr & vec_align) == 0 && (L.ldc & 3) == 0) ? 1 : 0;
    // C through TMA stores: {N, M}, row stride ldc * element bytes, 128-byte
    // swizzle, box 32 x 32 for FP32 and 64 x 32 for 16-bit types (128-byte
    // rows either way).  Needs a 16-byte aligned base and row stride.  The
    // store clips a box at C's last column only to a 16-byte boundary, so it
    // is used only when rows end on one (N a multiple of 4 FP32 or 8 16-bit
    // elements): otherwise the columns between N and the boundary -- the
    // caller's padding -- would be written.
    CUtensorMap map_c;
    memset(&map_c, 0, sizeof(map_c));
    a.tma_store = 0;
    const int ces = c_elem_bytes(L.ct);
    const int64_t row_quantum = 16 / ces;   // elements per 16 bytes
    if (!L.swap && (c_addr & 15) == 0 && (L.ldc % row_quantum) == 0 && (L.N % row_quantum) == 0) {
        const cuuint64_t dims[2] = {static_cast<cuuint64_t>(L.N), static_cast<cuuint64_t>(L.M)};
        const cuuint64_t strides[1] = {static_cast<cuuint64_t>(L.ldc) * ces};
        const cuuint32_t box[2] = {static_cast<cuuint32_t>(128 / ces), 32};
        const cuuint32_t estr[2] = {1, 1};
        const CUtensorMapDataType ty = L.ct == kCF32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                       : L.ct == kCF16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16
                                                       : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
        if (encode(&map_c, ty, 2, L.C, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS)
            a.tma_store = (L.store_mode == 1) ? 0 : 1;
    }
    a.p_kmajor = L.swap ? b_kmajor : a_kmajor;
    a.q_kmajor = L.swap ? a_kmajor : b_kmajor;
    // operand format code within the MMA kind
    const uint32_t fcode = L.fmt == 0 ? 0u : L.fmt == 1 ? 1u : L.fmt == 2 ? 2u : L.fmt == 3 ? 0u : 1u;
    a.idesc = idesc_f16_f32(fcode, !a.p_kmajor, !a.q_kmajor, L.pair ? 2 * kTcBM : kTcBM,
                            static_cast<uint32_t>(L.bn));
    a.ws = L.ws;
    a.counters = L.counters;
    a.ab = L.ab;
    a.alpha = L.alpha;
    a.beta = L.beta;
    a.wait_limit_ns = L.wait_limit_ns ? L.wait_limit_ns : kWaitLimitNs;
    a.stall_cta = L.stall_fill > 0 ? L.stall_cta : -1;
    a.stall_fill = L.stall_fill - 1;

    const CUtensorMap& mp = L.swap ? map_b : map_a;
    const CUtensorMap& mq = L.swap ? map_a : map_b;
    switch (tc_kind(L.fmt)) {
        case 0: return dispatch_kind<0>(L, map_a, map_b, mp, mq, map_c, a, stream);
        case 1: return dispatch_kind<1>(L, map_a, map_b, mp, mq, map_c, a, stream);
        case 2: return dispatch_kind<2>(L, map_a, map_b, mp, mq, map_c, a, stream);
    }
    return cudaErrorInvalidValue;
}

}  // namespace gb300
