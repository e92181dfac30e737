// api.cu -- the C ABI declared in include/gb300gemm.h: argument checks,
// planning, the split-K workspace and kernel launches.
//
// The operation and its conventions (row-major, leading dimension = row
// stride in elements, C overwritten) are those of the header; see there for
// the page passages they follow.

#include <algorithm>
#include <atomic>
#include <climits>
#include <cstdio>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>

#include "../../include/gb300gemm.h"
#include "cstore.cuh"
#include "internal.h"

using namespace gb300;

namespace {

thread_local char t_last_error[256] = "";
thread_local int64_t t_launches = 0;
std::atomic<int64_t> g_allocs{0};   // device allocations made by the library (all threads)

void note_cuda_error(cudaError_t e, const char* where) {
    snprintf(t_last_error, sizeof(t_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
             cudaGetErrorString(e));
}

// ---- device facts --------------------------------------------------------------

struct DeviceInfo {
    bool valid = false;
    int major = 0, minor = 0, sms = 0;
};

std::mutex g_dev_mu;
std::map<int, DeviceInfo> g_dev;

gemm_status_t current_device(int* dev, DeviceInfo* info) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetDevice");
        return GEMM_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_dev_mu);
    DeviceInfo& d = g_dev[*dev];
    if (!d.valid) {
        cudaDeviceProp p;
        e = cudaGetDeviceProperties(&p, *dev);
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaGetDeviceProperties");
            return GEMM_ERR_CUDA;
        }
        d.major = p.major;
        d.minor = p.minor;
        d.sms = p.multiProcessorCount;
        d.valid = true;
    }
    *info = d;
    if (d.major != 10 || d.minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
    return GEMM_OK;
}

// Most CTA-pair clusters (256-wide tiles) resident at once on the current
// device; 0 if the query fails (the pair kernel is then not planned).
int pair_clusters() {
    static std::mutex mu;
    static int cache[64];
    static bool known[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lk(mu);
    if (!known[dev]) {
        int n = 0;
        if (tc_pair_max_clusters(256, &n) != cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cache[dev] = n;
        known[dev] = true;
    }
    return cache[dev];
}

// Resident SGEMM CTAs on the whole device for a tile shape, micro-tile width
// and kernel form (split or stream-K), cached per device.
int sgemm_slots(int bm, int bn, int sms, bool stream_k = false, int tn = 8) {
    static std::mutex mu;
    static int cache[64][8];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    const int shape = tn == 16 ? 3 : (bm == 128 && bn == 128) ? 0 : (bm == 128 ? 1 : 2);
    const int idx = shape + (stream_k ? 4 : 0);
    std::lock_guard<std::mutex> lk(mu);
    if (!cache[dev][idx]) {
        int n = 0;
        if (sgemm_blocks_per_sm(bm, bn, tn, stream_k, &n) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
        cache[dev][idx] = n;
    }
    return cache[dev][idx] * sms;
}

EncodeTiledFn encode_fn() {
    static std::once_flag once;
    static EncodeTiledFn fn = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// ---- the current CUDA context ---------------------------------------------------
//
// Device pointers and stream handles the library caches belong to the CUDA
// context that was current when they were made.  cudaDeviceReset destroys
// the device's primary context (and every allocation in it); the next call
// then runs in a new context, where a cached pointer would be invalid.  So
// caches record the context's unique id (cuCtxGetId) and are dropped, not
// freed, when it changes.

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id (+1) of the context current on this thread, making the device's
// primary context current first if none is; 0 if it cannot be told.
uint64_t current_ctx_id(int dev) {
    static std::once_flag once;
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess && q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return 0;
    for (int attempt = 0; attempt < 2; ++attempt) {
        CUcontext c = nullptr;
        unsigned long long id = 0;
        if (get_current(&c) == CUDA_SUCCESS && c && get_id(c, &id) == CUDA_SUCCESS)
            return static_cast<uint64_t>(id) + 1;
        // no context current, or one that a reset has destroyed: cudaSetDevice
        // initialises the device's primary context and makes it current
        if (attempt == 0 && cudaSetDevice(dev) != cudaSuccess) {
            cudaGetLastError();
            return 0;
        }
    }
    return 0;
}

// ---- split-K workspace, one per (device, stream) --------------------------------

struct Workspace {
    float* ws = nullptr;
    size_t ws_floats = 0;
    uint32_t* counters = nullptr;
    size_t n_counters = 0;
    uint64_t ctx = 0;     // context the buffers belong to
    uint64_t epoch = 0;   // g_ws_epoch[dev] when the counters were last known to be zero
};

std::mutex g_ws_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;
// Per device: bumped each time gemm_device_error finds that a kernel gave up
// a wait.  A kernel that aborts may leave tile counters part-way, so every
// workspace of the device clears its counters before its next use.
std::map<int, uint64_t> g_ws_epoch;

gemm_status_t get_workspace(int dev, cudaStream_t stream, size_t floats, size_t counters,
                            float** ws, uint32_t** cnt) {
    const uint64_t ctx = current_ctx_id(dev);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    Workspace& w = g_ws[{dev, stream}];
    if (ctx && w.ctx != ctx) {
        // made in a context that no longer exists (or none yet): forget it
        w = Workspace{};
        w.ctx = ctx;
    }
    const uint64_t epoch = g_ws_epoch[dev];
    if (w.ws_floats < floats) {
        if (w.ws) {
            cudaStreamSynchronize(stream);   // the old buffer may still be in use on this stream
            cudaFree(w.ws);
            w.ws = nullptr;
            w.ws_floats = 0;
        }
        cudaError_t e = cudaMalloc(&w.ws, floats * sizeof(float));
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaMalloc(split-K workspace)");
            w.ws = nullptr;
            return GEMM_ERR_OUT_OF_MEMORY;
        }
        ++g_allocs;
        w.ws_floats = floats;
    }
    if (w.n_counters < counters) {
        if (w.counters) {
            cudaStreamSynchronize(stream);
            cudaFree(w.counters);
            w.counters = nullptr;
            w.n_counters = 0;
        }
        cudaError_t e = cudaMalloc(&w.counters, counters * sizeof(uint32_t));
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaMalloc(split-K counters)");
            w.counters = nullptr;
            return GEMM_ERR_OUT_OF_MEMORY;
        }
        ++g_allocs;
        w.n_counters = counters;
        w.epoch = epoch + 1;   // cleared below
    }
    // Counters start at zero and every completed launch leaves them at zero;
    // after a reported timeout (or when new) they are cleared on the stream.
    if (w.epoch != epoch) {
        cudaError_t e = cudaMemsetAsync(w.counters, 0, w.n_counters * sizeof(uint32_t), stream);
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaMemsetAsync(split-K counters)");
            return GEMM_ERR_CUDA;
        }
        w.epoch = epoch;
    }
    *ws = w.ws;
    *cnt = w.counters;
    return GEMM_OK;
}

// ---- argument checks -------------------------------------------------------------

// dtype codes of gemm_options_t: 0 FP16, 1 BF16, 2 FP32 (CUDA cores), 3 TF32
// (FP32 storage, tensor cores), 4 E4M3, 5 E5M2.
int dtype_bytes(int dtype) { return dtype <= 1 ? 2 : dtype <= 3 ? 4 : 1; }
int tc_fmt_of(int dtype) { return dtype <= 1 ? dtype : dtype - 1; }

bool spans_overlap(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) {
    return a0 < b1 && b0 < a1;
}

gemm_status_t check_args(const void* A, const void* B, const void* C, int64_t M, int64_t N,
                         int64_t K, int64_t lda, int64_t ldb, int64_t ldc, int esize,
                         int trans_a = 0, int trans_b = 0, int c_dtype = 0) {
    if (c_dtype < 0 || c_dtype > 2) return GEMM_ERR_INVALID_VALUE;
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_VALUE;
    if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_INVALID_VALUE;
    if (trans_a < 0 || trans_a > 1 || trans_b < 0 || trans_b > 1) return GEMM_ERR_INVALID_VALUE;
    // stored shapes: A is M x K (or K x M transposed), B is K x N (or N x K)
    const int64_t a_rows = trans_a ? K : M, a_cols = trans_a ? M : K;
    const int64_t b_rows = trans_b ? N : K, b_cols = trans_b ? K : N;
    if (lda < a_cols || ldb < b_cols || ldc < N) return GEMM_ERR_INVALID_VALUE;
    if (M == 0 || N == 0) return GEMM_OK;
    if (!C) return GEMM_ERR_INVALID_VALUE;
    if (K > 0 && (!A || !B)) return GEMM_ERR_INVALID_VALUE;
    // keep every byte offset well inside int64
    const int64_t lim = INT64_MAX / 16;
    if ((M > 1 && ldc > lim / (M - 1)) || (a_rows > 1 && lda > lim / (a_rows - 1)) ||
        (b_rows > 1 && ldb > lim / (b_rows - 1)))
        return GEMM_ERR_INVALID_VALUE;
    const uintptr_t c0 = reinterpret_cast<uintptr_t>(C);
    const uintptr_t c1 = c0 + static_cast<uintptr_t>((M - 1) * ldc + N) * c_elem_bytes(c_dtype);
    if (K > 0) {
        const uintptr_t a0 = reinterpret_cast<uintptr_t>(A);
        const uintptr_t a1 = a0 + static_cast<uintptr_t>((a_rows - 1) * lda + a_cols) * esize;
        const uintptr_t b0 = reinterpret_cast<uintptr_t>(B);
        const uintptr_t b1 = b0 + static_cast<uintptr_t>((b_rows - 1) * ldb + b_cols) * esize;
        if (spans_overlap(c0, c1, a0, a1) || spans_overlap(c0, c1, b0, b1)) return GEMM_ERR_OVERLAP;
    }
    return GEMM_OK;
}

// ---- planning ----------------------------------------------------------------------

enum class Kind { Nothing, ZeroFill, Tc, Generic, Sgemm };

struct Plan {
    Kind kind = Kind::Nothing;
    int ab = 0;              // 0: C = AB; 1: alpha AB; 2: alpha AB + beta C
    float alpha = 1.0f, beta = 0.0f;
    int trans_a = 0, trans_b = 0;
    int ct = 0;              // C's type (cstore.cuh)
    TcLaunch tc{};
    SgemmLaunch sg{};
    int64_t units = 0;
    size_t ws_floats = 0, n_counters = 0;
};

gemm_status_t make_plan(int dtype, const void* A, const void* B, void* C, int64_t M, int64_t N,
                        int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                        const gemm_options_t& o, int sms, Plan* plan) {
    Plan p;
    if (o.epilogue < 0 || o.epilogue > 1) return GEMM_ERR_INVALID_VALUE;
    if (o.trans_a < 0 || o.trans_a > 1 || o.trans_b < 0 || o.trans_b > 1) return GEMM_ERR_INVALID_VALUE;
    p.trans_a = o.trans_a;
    p.trans_b = o.trans_b;
    if (o.c_dtype < 0 || o.c_dtype > 2) return GEMM_ERR_INVALID_VALUE;
    p.ct = o.c_dtype;
    if (o.epilogue) {
        p.alpha = o.alpha;
        p.beta = o.beta;
        p.ab = (p.beta != 0.0f) ? 2 : (p.alpha != 1.0f ? 1 : 0);
    }
    if (M == 0 || N == 0) {
        *plan = p;
        return GEMM_OK;
    }
    if (K == 0) {
        p.kind = Kind::ZeroFill;
        *plan = p;
        return GEMM_OK;
    }
    if (dtype == 2) {
        // float4 operand loads; C stores of 4 elements (16 bytes FP32, 8 bytes 16-bit)
        const uintptr_t c_align = p.ct == 0 ? 15 : 7;
        const bool aligned = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15) == 0 &&
                             (reinterpret_cast<uintptr_t>(C) & c_align) == 0 &&
                             (lda & 3) == 0 && (ldb & 3) == 0 && (ldc & 3) == 0;
        if (o.generic || !aligned || o.trans_a || o.trans_b) {
            p.kind = Kind::Generic;
        } else {
            p.kind = Kind::Sgemm;
            SgemmLaunch& S = p.sg;
            S.ab = p.ab;
            S.alpha = p.alpha;
            S.beta = p.beta;
            S.A = static_cast<const float*>(A);
            S.B = static_cast<const float*>(B);
            S.C = C;
            S.ct = p.ct;
            S.M = M; S.N = N; S.K = K; S.lda = lda; S.ldb = ldb; S.ldc = ldc;
            if (o.stream_k < 0 || o.stream_k > 2) return GEMM_ERR_INVALID_VALUE;
            const int bk = sgemm_k_step();
            const int64_t kb = ceil_div(K, bk);
            // Stream-K by default when it balances better than whole waves of
            // tiles (measured from 512^3 to 8192^3, see sgemm.cu): below 3
            // waves of 128 x 128 tiles it beat the split plans by 5-29 %; the
            // tile is the largest whose persistent CTAs still get enough K
            // steps each (128 x 128 from 32, 128 x 64 from 8, else 64 x 64).
            // From 3 waves on, whole waves of 128 x 128 tiles with 8 x 16
            // outputs per thread (128 threads) were 1-5 % faster than both
            // (4096^3 to 8192^3, 16384 x 4096 x 4096, 8192 x 8192 x 2048).
            bool auto_sk = false, auto_wide = false;
            int sk_bm = 128, sk_bn = 64;
            if (o.stream_k == 0 && o.split_k <= 0 && o.tile_n == 0 && M > 64) {
                const int64_t s128 = sgemm_slots(128, 128, sms, true);
                const int64_t s64 = sgemm_slots(128, 64, sms, true);
                if (s128 > 0 && s64 > 0) {
                    const int64_t t128 = ceil_div(M, 128) * ceil_div(N, 128);
                    const int64_t t64 = ceil_div(M, 128) * ceil_div(N, 64);
                    if (t128 < 3 * s128) {
                        auto_sk = true;
                        if (N > 64 && t128 * kb >= 32 * s128) {
                            sk_bn = 128;
                        } else if (t64 * kb < 8 * s64) {
                            sk_bm = 64;
                        }
                    } else if (N > 64) {
                        auto_wide = true;
                    }
                }
            }
            // With 8 x 8 outputs per thread, 128 x 64 tiles measured faster
            // than 128 x 128 from 2048^3 to 8192 x 8192 x 2048 (3 CTAs of 4
            // warps per SM against 2 of 8).
            S.tn = 8;
            if (auto_sk) {
                S.bm = sk_bm; S.bn = sk_bn;
            } else if (o.tile_n == 256 || auto_wide) {   // 128 x 128 tiles, 8 x 16 per thread
                S.bm = 128; S.bn = 128; S.tn = 16;
            } else if (o.tile_n == 128) {
                S.bm = 128; S.bn = 128;
            } else if (o.tile_n == 64 || (o.tile_n == 0 && M > 64)) {
                S.bm = 128; S.bn = 64;
            } else if (o.tile_n == 0 || o.tile_n == 32) {
                S.bm = 64; S.bn = 64;
            } else {
                return GEMM_ERR_INVALID_VALUE;
            }
            if (o.split_k < 0 || o.split_k > 64) return GEMM_ERR_INVALID_VALUE;
            const int64_t tiles = ceil_div(M, S.bm) * ceil_div(N, S.bn);
            const int64_t slots = static_cast<int64_t>(sgemm_slots(S.bm, S.bn, sms, false, S.tn));
            auto part = [&](int64_t t0, int64_t nt, int64_t splits) {
                splits = std::max<int64_t>(1, std::min<int64_t>(splits, kb));
                const int64_t chunk = ceil_div(ceil_div(K, splits), bk) * bk;
                splits = ceil_div(K, chunk);   // no empty slices
                SgemmPart& q = S.parts[S.nparts++];
                q.tile0 = static_cast<int>(t0);
                q.tiles = static_cast<int>(nt);
                q.splits = static_cast<int>(splits);
                q.k_chunk = static_cast<int>(chunk);
                if (splits > 1) {
                    p.ws_floats = std::max<size_t>(p.ws_floats, static_cast<size_t>(nt * splits * S.bm * S.bn));
                    p.n_counters = std::max<size_t>(p.n_counters, static_cast<size_t>(nt));
                }
            };
            S.nparts = 0;
            const int64_t sk_slots = static_cast<int64_t>(sgemm_slots(S.bm, S.bn, sms, true, S.tn));
            if (o.split_k <= 0 && (o.stream_k == 2 || auto_sk) && sk_slots > 0) {
                // Stream-K: a persistent grid of the resident CTAs takes whole
                // tiles while whole waves last, then shares the remaining
                // tiles' K steps out evenly (cut tiles summed in piece order).
                int64_t G = sk_slots;
                int64_t dp = 0;
                if (tiles >= G) dp = (tiles % G == 0) ? tiles : (tiles / G - 1) * G;
                const int64_t W = (tiles - dp) * kb;
                if (W > 0 && W < G) G = W;
                if (W == 0) G = std::min<int64_t>(G, tiles);
                SgemmPart& q = S.parts[S.nparts++];
                q.tile0 = 0;
                q.tiles = static_cast<int>(tiles);
                q.splits = 1;
                q.k_chunk = static_cast<int>(kb * bk);
                q.sk_mode = 1;
                q.dp_tiles = static_cast<int>(dp);
                q.sk_kblocks = W;
                q.grid = static_cast<int>(std::max<int64_t>(G, 1));
                int max_seg = 1;
                const int64_t sk_tiles = tiles - dp;
                for (int64_t ts = 0; ts < sk_tiles && W > 0; ++ts) {
                    const int64_t first = ((ts * kb + 1) * G - 1) / W;
                    const int64_t last = (((ts + 1) * kb) * G - 1) / W;
                    max_seg = std::max<int>(max_seg, static_cast<int>(last - first + 1));
                }
                q.max_seg = max_seg;
                if (max_seg > 1) {
                    p.ws_floats = static_cast<size_t>(sk_tiles * max_seg * S.bm * S.bn);
                    p.n_counters = static_cast<size_t>(sk_tiles);
                }
                p.units = tiles;
                *plan = p;
                return GEMM_OK;
            }
            if (o.split_k > 0) {
                part(0, tiles, o.split_k);
            } else if (slots > 0 && tiles >= slots) {
                // Whole waves as they are; a short last wave is split along K so
                // that it occupies more CTAs for less time.
                const int64_t waves = tiles / slots;
                const int64_t tail = tiles - waves * slots;
                const int64_t s_tail = std::min<int64_t>({4, tail ? slots / tail : 1, kb / 16});
                if (tail > 0 && 2 * tail <= slots && s_tail >= 2) {
                    part(0, waves * slots, 1);
                    part(waves * slots, tail, s_tail);
                } else {
                    part(0, tiles, 1);
                }
            } else if (slots > 0) {
                // Fewer tiles than resident CTAs: split K to fill the GPU.
                part(0, tiles, std::min<int64_t>({8, slots / std::max<int64_t>(tiles, 1), kb / 16}));
            } else {
                part(0, tiles, 1);
            }
            p.units = 0;
            for (int i = 0; i < S.nparts; ++i) p.units += static_cast<int64_t>(S.parts[i].tiles) * S.parts[i].splits;
        }
        *plan = p;
        return GEMM_OK;
    }

    // Tensor-core inputs: TMA needs 16-byte aligned bases and row strides.
    const int es = dtype_bytes(dtype);
    const bool tma_ok = ((reinterpret_cast<uintptr_t>(A) | reinterpret_cast<uintptr_t>(B)) & 15) == 0 &&
                        (lda * es) % 16 == 0 && (ldb * es) % 16 == 0;
    if (dtype >= 3) {
        // TF32 and 8-bit inputs run only on the tensor cores, with both
        // operands K-contiguous: A stored M x K, B stored N x K.
        if (o.generic || !tma_ok || o.trans_a || !o.trans_b) return GEMM_ERR_INVALID_VALUE;
    } else if (o.generic || !tma_ok) {
        p.kind = Kind::Generic;
        *plan = p;
        return GEMM_OK;
    }
    TcLaunch& L = p.tc;
    L.trans_a = p.trans_a;
    L.trans_b = p.trans_b;
    L.ab = p.ab;
    L.alpha = p.alpha;
    L.beta = p.beta;
    L.A = A; L.B = B; L.C = C;
    L.ct = p.ct;
    L.M = M; L.N = N; L.K = K; L.lda = lda; L.ldb = ldb; L.ldc = ldc;
    L.fmt = tc_fmt_of(dtype);
    // swap-AB for small M -- unless CTA pairs were asked for, which never swap
    L.swap = (o.swap_ab < 0) ? ((M <= 64 && N > M && o.cta_pair != 2) ? 1 : 0) : (o.swap_ab ? 1 : 0);
    if (o.cta_pair < 0 || o.cta_pair > 2) return GEMM_ERR_INVALID_VALUE;
    if (o.store_mode < 0 || o.store_mode > 1) return GEMM_ERR_INVALID_VALUE;
    if (o.stream_k < 0 || o.stream_k > 3) return GEMM_ERR_INVALID_VALUE;
    L.store_mode = o.store_mode;

    // CTA pairs: two SMs share a 256-row tile (each loads half the operand
    // bytes a 128-row tile would).  Chosen when there are at least 80 % of a
    // full wave of such tiles and no split-K is asked for (2048^3: 64 pair
    // tiles on 76 clusters run 3.6 % faster than 128 one-CTA 128 x 256 tiles;
    // 1024^3, 16 pair tiles, ran 42 % slower than one-CTA 128 x 64 tiles).
    if (o.cta_pair == 2 || (o.cta_pair == 0 && !L.swap && o.split_k <= 1 && M >= 256 &&
                            N >= 256 && K >= 512 && (o.tile_n == 0 || o.tile_n == 256))) {
        const int max_cl = pair_clusters();
        const int bn = o.tile_n ? o.tile_n : 256;
        const int64_t units = ceil_div(M, 2 * kTcBM) * ceil_div(N, bn);
        const bool forced = o.cta_pair == 2;
        if (forced && (L.swap || o.split_k > 1 || !tc_config_supported(bn, 0, 1) || max_cl < 1))
            return GEMM_ERR_INVALID_VALUE;
        if (max_cl >= 1 && (forced || 5 * units >= 4 * static_cast<int64_t>(max_cl))) {
            L.pair = 1;
            L.bn = bn;
            L.splits = 1;
            int64_t group = o.group_m > 0 ? o.group_m : 8;
            const int64_t tiles_p = ceil_div(M, 2 * kTcBM);
            if (group > tiles_p) group = tiles_p;
            L.group = static_cast<int>(group);
            const int64_t clusters = std::min<int64_t>(units, max_cl);
            L.grid = static_cast<int>(2 * clusters);
            p.units = units;
            // Stream-K on request only.  Measured at 4096^3 and 8192^3 (BF16
            // and E4M3) it is 2-6 % slower than whole tiles: the kernel runs
            // at the power cap, so the clusters left idle by a partial last
            // wave let the busy ones clock higher, while the partial sums'
            // workspace traffic costs energy.
            const int64_t ksteps = ceil_div(K, static_cast<int64_t>(tc_k_elems(L.fmt)) * kPairAtoms);
            // Tail split by default once there are at least 8 whole waves:
            // the tiles left after the last whole wave are cut into equal K
            // pieces over more clusters.  At 8192^3 (13 waves + 36 tiles) it
            // measured +1.3 % best-of-10, +0.8 % in 100-launch loops and
            // +0.5 % over 3 s at the power cap; at 4096^3 (3 waves + 28) it
            // lost 2.5 %, the pieces' round trip weighing more on 3 waves.
            const bool auto_tail = o.stream_k == 0 && units >= 8 * clusters && units % clusters != 0 &&
                                   2 * (units % clusters) <= clusters;
            if (o.stream_k == 2 || o.stream_k == 3 || auto_tail) {
                const int64_t slot_tiles =
                    o.stream_k == 2 ? tc_streamk_schedule(L, units, ksteps, static_cast<int>(clusters))
                                    : tc_tailsplit_schedule(L, units, ksteps, static_cast<int>(clusters));
                L.grid *= 2;   // the schedule counts clusters
                if (slot_tiles > 0) {
                    p.ws_floats = static_cast<size_t>(slot_tiles * L.max_seg * 2 * kTcBM * L.bn);
                    p.n_counters = static_cast<size_t>(slot_tiles * 8);
                }
            }
            p.kind = Kind::Tc;
            *plan = p;
            return GEMM_OK;
        }
    }

    const int64_t pe = L.swap ? N : M;     // extent along the MMA M side
    const int64_t qe = L.swap ? M : N;     // extent along the MMA N side
    if (o.tile_n) {
        if (!tc_config_supported(o.tile_n, L.swap, 0)) return GEMM_ERR_INVALID_VALUE;
        if (L.swap && L.trans_a && o.tile_n % 64) return GEMM_ERR_INVALID_VALUE;
        L.bn = o.tile_n;
    } else if (L.swap) {
        // with A stored transposed the swapped B operand (rows of C) is
        // M-contiguous, loaded in 64-row boxes: BN = 64
        L.bn = L.trans_a ? 64 : (qe <= 16 ? 16 : qe <= 32 ? 32 : 64);
    } else if (qe <= 64) {
        L.bn = 64;
    } else {
        // fewest estimated tile-time units: waves x (tile width + fixed cost)
        const int cand[3] = {256, 128, 64};
        int64_t best = INT64_MAX;
        for (int bn : cand) {
            if (bn > 128 && qe <= 128) continue;
            const int64_t tiles = ceil_div(pe, kTcBM) * ceil_div(qe, bn);
            const int64_t cost = ceil_div(tiles, sms) * (bn + 64);
            if (cost < best) {
                best = cost;
                L.bn = bn;
            }
        }
    }
    const int64_t tiles_p = ceil_div(pe, kTcBM);
    const int64_t tiles = tiles_p * ceil_div(qe, L.bn);
    const int64_t kb_total = ceil_div(K, tc_k_elems(L.fmt));

    int64_t group = o.group_m > 0 ? o.group_m : 16;
    if (group > tiles_p) group = tiles_p;
    L.group = static_cast<int>(group);

    if (o.split_k <= 0 && (o.stream_k == 2 || o.stream_k == 3)) {
        // Stream-K: whole tiles while whole waves last, then the remaining
        // tiles' k-blocks shared evenly by every CTA (partial tiles summed in
        // a fixed order), so no SM idles through a partial last wave.  Opt-in:
        // on the measured shapes it is slower than whole tiles, and a variant
        // that moves no partial sums at all is still no faster.
        const int64_t slot_tiles = o.stream_k == 2 ? tc_streamk_schedule(L, tiles, kb_total, sms)
                                                   : tc_tailsplit_schedule(L, tiles, kb_total, sms);
        p.units = tiles;
        if (slot_tiles > 0) {
            p.ws_floats = static_cast<size_t>(slot_tiles * L.max_seg * kTcBM * L.bn);
            p.n_counters = static_cast<size_t>(slot_tiles * 4);
        }
        p.kind = Kind::Tc;
        *plan = p;
        return GEMM_OK;
    }

    int64_t splits = 1;
    if (o.split_k > 0) {
        if (o.split_k > 64) return GEMM_ERR_INVALID_VALUE;
        splits = o.split_k;
    } else if (tiles * 2 <= sms && kb_total >= 4) {
        // few tiles: split K so that more SMs stream operands.  Minimise
        // waves x (1/S + a fixed cost per unit).
        double best = 1e30;
        const int64_t smax = std::min<int64_t>(16, kb_total / 2);
        for (int64_t s = 1; s <= smax; ++s) {
            const double cost = static_cast<double>(ceil_div(tiles * s, sms)) * (1.0 / s + 0.05);
            if (cost < best - 1e-12) {
                best = cost;
                splits = s;
            }
        }
    }
    if (splits > kb_total) splits = kb_total;
    const int64_t kb_per = ceil_div(kb_total, splits);
    splits = ceil_div(kb_total, kb_per);   // no empty slices
    L.splits = static_cast<int>(splits);
    L.max_seg = L.splits;

    p.units = tiles * splits;
    L.grid = static_cast<int>(std::min<int64_t>(p.units, sms));
    if (splits > 1) {
        p.ws_floats = static_cast<size_t>(tiles * splits * kTcBM * L.bn);
        p.n_counters = static_cast<size_t>(tiles * 4);
    }
    p.kind = Kind::Tc;
    *plan = p;
    return GEMM_OK;
}

void describe_kernel(const Plan& p, int dtype, char* buf, int n);

const char* fmt_name(int fmt) {
    static const char* names[] = {"f16", "bf16", "tf32", "e4m3", "e5m2"};
    return (fmt >= 0 && fmt <= 4) ? names[fmt] : "?";
}

void describe(const Plan& p, int dtype, char* buf, int64_t size) {
    if (!buf || size <= 0) return;
    const int n = static_cast<int>(size > INT32_MAX ? INT32_MAX : size);
    describe_kernel(p, dtype, buf, n);
    if (p.ab) {
        const size_t len = strlen(buf);
        if (static_cast<int64_t>(len) + 1 < n)
            snprintf(buf + len, n - len, " epilogue=%s alpha=%g beta=%g",
                     p.ab == 2 ? "alpha*AB+beta*C" : "alpha*AB", p.alpha, p.beta);
    }
    if (p.ct) {
        const size_t len = strlen(buf);
        if (static_cast<int64_t>(len) + 1 < n)
            snprintf(buf + len, n - len, " c=%s", p.ct == 1 ? "f16" : "bf16");
    }
}

void describe_kernel(const Plan& p, int dtype, char* buf, int n) {
    switch (p.kind) {
        case Kind::Nothing: snprintf(buf, n, "nothing (empty output)"); break;
        case Kind::ZeroFill: snprintf(buf, n, "zero-fill (K == 0)"); break;
        case Kind::Generic: snprintf(buf, n, "generic cuda-core dtype=%d tile=64x64", dtype); break;
        case Kind::Sgemm: {
            const SgemmPart& a = p.sg.parts[0];
            if (a.sk_mode)
                snprintf(buf, n, "sgemm tile=%dx%dx%d%s stream_k tiles=%d dp_tiles=%d sk_kblocks=%lld "
                         "max_seg=%d grid=%d", p.sg.bm, p.sg.bn, sgemm_k_step(),
                         p.sg.tn == 16 ? " thread=8x16" : "", a.tiles, a.dp_tiles,
                         static_cast<long long>(a.sk_kblocks), a.max_seg, a.grid);
            else if (p.sg.nparts == 1)
                snprintf(buf, n, "sgemm tile=%dx%dx%d%s tiles=%d split_k=%d units=%lld", p.sg.bm,
                         p.sg.bn, sgemm_k_step(), p.sg.tn == 16 ? " thread=8x16" : "", a.tiles, a.splits,
                         static_cast<long long>(p.units));
            else
                snprintf(buf, n, "sgemm tile=%dx%dx%d%s tiles=%d+%d split_k=%d+%d units=%lld",
                         p.sg.bm, p.sg.bn, sgemm_k_step(), p.sg.tn == 16 ? " thread=8x16" : "", a.tiles,
                         p.sg.parts[1].tiles, a.splits,
                         p.sg.parts[1].splits, static_cast<long long>(p.units));
            break;
        }
        case Kind::Tc:
            if (p.tc.sk_mode)
                snprintf(buf, n,
                         "tcgen05 fmt=%s tile=%dx%d pair=%d swap=%d %s dp_tiles=%d sk_kblocks=%lld "
                         "max_seg=%d group=%d units=%lld grid=%d",
                         fmt_name(p.tc.fmt), p.tc.pair ? 256 : 128, p.tc.bn, p.tc.pair,
                         p.tc.swap, p.tc.sk_ctas ? "tail_split" : "stream_k", p.tc.dp_tiles,
                         static_cast<long long>(p.tc.sk_kblocks),
                         p.tc.max_seg, p.tc.group, static_cast<long long>(p.units), p.tc.grid);
            else
                snprintf(buf, n,
                         "tcgen05 fmt=%s tile=%dx%d pair=%d swap=%d split_k=%d group=%d units=%lld grid=%d",
                         fmt_name(p.tc.fmt), p.tc.pair ? 256 : 128, p.tc.bn, p.tc.pair,
                         p.tc.swap, p.tc.splits, p.tc.group, static_cast<long long>(p.units), p.tc.grid);
            break;
    }
}

gemm_status_t launch_status(cudaError_t e, const char* what) {
    if (e == cudaSuccess) {
        ++t_launches;
        return GEMM_OK;
    }
    note_cuda_error(e, what);
    cudaGetLastError();   // clear a non-sticky launch error
    return GEMM_ERR_LAUNCH;
}

// A self-test of the tensor-core kernels' bounded waits (gemm_ex_stall_selftest).
struct StallTest {
    uint64_t limit_ns;
    int cta, fill;
};

gemm_status_t run(int dtype, const void* A, const void* B, void* C, int64_t M, int64_t N,
                  int64_t K, int64_t lda, int64_t ldb, int64_t ldc, const gemm_options_t& o,
                  cudaStream_t stream, const StallTest* stall = nullptr) {
    if (dtype < 0 || dtype > 5) return GEMM_ERR_INVALID_VALUE;
    const int esize = dtype_bytes(dtype);
    gemm_status_t st = check_args(A, B, C, M, N, K, lda, ldb, ldc, esize, o.trans_a, o.trans_b,
                                  o.c_dtype);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev;
    DeviceInfo info;
    st = current_device(&dev, &info);
    if (st != GEMM_OK) return st;
    Plan p;
    st = make_plan(dtype, A, B, C, M, N, K, lda, ldb, ldc, o, info.sms, &p);
    if (st != GEMM_OK) return st;
    if (stall) {
        // only the tensor-core kernels have pipeline waits; the stalled CTA
        // (pair kernel: cluster) must exist
        const int units = p.tc.pair ? p.tc.grid / 2 : p.tc.grid;
        if (p.kind != Kind::Tc || stall->cta < 0 || stall->cta >= units || stall->fill < 0) {
            snprintf(t_last_error, sizeof(t_last_error),
                     "stall self-test needs a tensor-core plan, 0 <= stall_cta < %d, stall_fill >= 0",
                     p.kind == Kind::Tc ? units : 0);
            return GEMM_ERR_INVALID_VALUE;
        }
        p.tc.wait_limit_ns = stall->limit_ns;
        p.tc.stall_cta = stall->cta;
        p.tc.stall_fill = stall->fill + 1;
    }
    switch (p.kind) {
        case Kind::Nothing: return GEMM_OK;
        case Kind::ZeroFill:   // the empty sum: beta * C, or zeros
            return launch_status(fill_scale_launch(C, p.ct, M, N, ldc, p.ab == 2 ? p.beta : 0.0f, stream),
                                 "fill_scale");
        case Kind::Generic:
            return launch_status(generic_launch(dtype, A, B, C, p.ct, M, N, K, lda, ldb, ldc, p.ab, p.alpha,
                                                p.beta, p.trans_a, p.trans_b, stream),
                                 "generic_gemm");
        case Kind::Sgemm:
            if (p.ws_floats) {
                st = get_workspace(dev, stream, p.ws_floats, p.n_counters, &p.sg.ws, &p.sg.counters);
                if (st != GEMM_OK) return st;
            }
            return launch_status(sgemm_launch(p.sg, stream), "sgemm");
        case Kind::Tc: {
            EncodeTiledFn enc = encode_fn();
            if (!enc) {
                snprintf(t_last_error, sizeof(t_last_error),
                         "cuTensorMapEncodeTiled entry point unavailable");
                return GEMM_ERR_CUDA;
            }
            if (p.ws_floats) {
                st = get_workspace(dev, stream, p.ws_floats, p.n_counters, &p.tc.ws, &p.tc.counters);
                if (st != GEMM_OK) return st;
            }
            return launch_status(tc_gemm_launch(p.tc, enc, stream), "tc_gemm");
        }
    }
    return GEMM_ERR_INVALID_VALUE;
}

gemm_options_t default_options(int dtype) {
    gemm_options_t o;
    memset(&o, 0, sizeof(o));
    o.dtype = dtype;
    o.swap_ab = -1;
    return o;
}

}  // namespace

extern "C" {

gemm_status_t gemm_f16f32(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                          int64_t lda, int64_t ldb, int64_t ldc, gemm_stream_t stream) {
    return run(0, A, B, C, M, N, K, lda, ldb, ldc, default_options(0),
               reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_bf16f32(const void* A, const void* B, float* C, int64_t M, int64_t N, int64_t K,
                           int64_t lda, int64_t ldb, int64_t ldc, gemm_stream_t stream) {
    return run(1, A, B, C, M, N, K, lda, ldb, ldc, default_options(1),
               reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t sgemm_f32(const float* A, const float* B, float* C, int64_t M, int64_t N, int64_t K,
                        int64_t lda, int64_t ldb, int64_t ldc, gemm_stream_t stream) {
    return run(2, A, B, C, M, N, K, lda, ldb, ldc, default_options(2),
               reinterpret_cast<cudaStream_t>(stream));
}

static gemm_status_t run_bt(int dtype, const void* A, const void* Bt, void* C, int64_t M,
                            int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                            gemm_stream_t stream) {
    gemm_options_t o = default_options(dtype);
    o.trans_b = 1;
    return run(dtype, A, Bt, C, M, N, K, lda, ldb, ldc, o, reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_tf32f32_bt(const float* A, const float* Bt, float* C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream) {
    return run_bt(3, A, Bt, C, M, N, K, lda, ldb, ldc, stream);
}

gemm_status_t gemm_e4m3f32_bt(const void* A, const void* Bt, float* C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream) {
    return run_bt(4, A, Bt, C, M, N, K, lda, ldb, ldc, stream);
}

gemm_status_t gemm_e5m2f32_bt(const void* A, const void* Bt, float* C, int64_t M, int64_t N,
                              int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                              gemm_stream_t stream) {
    return run_bt(5, A, Bt, C, M, N, K, lda, ldb, ldc, stream);
}

gemm_status_t gemm_ex(const void* A, const void* B, void* C, int64_t M, int64_t N, int64_t K,
                      int64_t lda, int64_t ldb, int64_t ldc, const gemm_options_t* options,
                      gemm_stream_t stream) {
    if (!options) return GEMM_ERR_INVALID_VALUE;
    return run(options->dtype, A, B, C, M, N, K, lda, ldb, ldc, *options,
               reinterpret_cast<cudaStream_t>(stream));
}

gemm_status_t gemm_plan_describe(int32_t dtype, const void* A, const void* B, const void* C,
                                 int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                 int64_t ldc, const gemm_options_t* options, char* buf,
                                 int64_t size) {
    if (buf && size > 0) buf[0] = '\0';
    if (dtype < 0 || dtype > 5) return GEMM_ERR_INVALID_VALUE;
    gemm_options_t o = options ? *options : default_options(dtype);
    gemm_status_t st = check_args(A, B, C, M, N, K, lda, ldb, ldc, dtype_bytes(dtype), o.trans_a,
                                  o.trans_b, o.c_dtype);
    if (st != GEMM_OK) return st;
    int dev;
    DeviceInfo info;
    st = current_device(&dev, &info);
    if (st != GEMM_OK) return st;
    Plan p;
    st = make_plan(dtype, A, B, const_cast<void*>(C), M, N, K, lda, ldb, ldc, o, info.sms, &p);
    if (st == GEMM_OK) describe(p, dtype, buf, size);
    return st;
}

gemm_status_t gemm_device_error(gemm_stream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetDevice");
        return GEMM_ERR_CUDA;
    }
    e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaStreamSynchronize");
        return GEMM_ERR_CUDA;
    }
    uint32_t* word = nullptr;
    e = tc_error_word(&word);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetSymbolAddress");
        return GEMM_ERR_CUDA;
    }
    uint32_t v = 0;
    e = cudaMemcpy(&v, word, sizeof(v), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaMemcpy(error word)");
        return GEMM_ERR_CUDA;
    }
    if (v) {
        e = cudaMemset(word, 0, sizeof(uint32_t));
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaMemset(error word)");
            return GEMM_ERR_CUDA;
        }
        {
            // a kernel that gave up may have left split-K tile counters part-way:
            // every workspace of this device clears them before its next use
            std::lock_guard<std::mutex> lk(g_ws_mu);
            ++g_ws_epoch[dev];
        }
        snprintf(t_last_error, sizeof(t_last_error), "device pipeline wait gave up (bits 0x%x)", v);
        return GEMM_ERR_DEVICE_TIMEOUT;
    }
    return GEMM_OK;
}

gemm_status_t gemm_watchdog_selftest(int32_t limit_ms, gemm_stream_t stream) {
    if (limit_ms < 1 || limit_ms > 2000) return GEMM_ERR_INVALID_VALUE;
    int dev;
    DeviceInfo info;
    gemm_status_t st = current_device(&dev, &info);
    if (st != GEMM_OK) return st;
    return launch_status(watchdog_selftest_launch(static_cast<uint64_t>(limit_ms) * 1000000ull,
                                                  reinterpret_cast<cudaStream_t>(stream)),
                         "watchdog_selftest");
}

gemm_status_t gemm_release_workspace(void) {
    int dev;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetDevice");
        return GEMM_ERR_CUDA;
    }
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaDeviceSynchronize");
        return GEMM_ERR_CUDA;
    }
    const uint64_t ctx = current_ctx_id(dev);
    std::lock_guard<std::mutex> lk(g_ws_mu);
    for (auto it = g_ws.begin(); it != g_ws.end();) {
        if (it->first.first == dev) {
            if (!ctx || it->second.ctx == ctx) {   // else its context (and memory) is gone
                cudaFree(it->second.ws);
                cudaFree(it->second.counters);
            }
            it = g_ws.erase(it);
        } else {
            ++it;
        }
    }
    return GEMM_OK;
}

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_VALUE: return "GEMM_ERR_INVALID_VALUE: invalid argument";
        case GEMM_ERR_OVERLAP: return "GEMM_ERR_OVERLAP: C overlaps A or B";
        case GEMM_ERR_UNSUPPORTED_DEVICE: return "GEMM_ERR_UNSUPPORTED_DEVICE: needs compute capability 10.3";
        case GEMM_ERR_LAUNCH: return "GEMM_ERR_LAUNCH: kernel launch failed";
        case GEMM_ERR_DEVICE_TIMEOUT: return "GEMM_ERR_DEVICE_TIMEOUT: a device pipeline wait gave up";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA: CUDA runtime call failed";
        case GEMM_ERR_OUT_OF_MEMORY: return "GEMM_ERR_OUT_OF_MEMORY: workspace allocation failed";
    }
    return "unknown gemm_status_t";
}

const char* gemm_last_cuda_error(void) { return t_last_error; }

int32_t gemm_version(void) { return 200; }

int64_t gemm_launch_count(void) { return t_launches; }

int64_t gemm_alloc_count(void) { return g_allocs.load(); }

gemm_status_t gemm_ex_stall_selftest(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                     int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                     const gemm_options_t* options, int32_t limit_ms,
                                     int32_t stall_cta, int32_t stall_fill, gemm_stream_t stream) {
    if (!options || limit_ms < 1 || limit_ms > 2000) return GEMM_ERR_INVALID_VALUE;
    const StallTest t{static_cast<uint64_t>(limit_ms) * 1000000ull, stall_cta, stall_fill};
    return run(options->dtype, A, B, C, M, N, K, lda, ldb, ldc, *options,
               reinterpret_cast<cudaStream_t>(stream), &t);
}

}  // extern "C"

// ---- allocation-free entry point ------------------------------------------------
//
// gemm_ex_noalloc serves callers that must not allocate device memory after
// start-up: applications that hand the GPU's memory to their own pool and
// account for every byte, and latency-critical loops in which a cudaMalloc
// or cudaFree (which can synchronise the device) is not acceptable.  It runs
// the same kernels as gemm_ex; the only difference is where the split-K
// tensor-core kernel keeps its scratch (partial tiles and arrival counters):
// in the file-scope array below instead of a workspace allocated on first use.

namespace {

constexpr size_t kNoallocScratchBytes = GEMM_NOALLOC_SCRATCH_BYTES;
constexpr size_t kNoallocCounterBytes = 64 * 1024;   // counters for up to 4096 tiles
constexpr int kNoallocMaxDevices = 64;

// Every device that loads this library holds this array until the process
// exits.  In host code the name is only a stand-in: its device address comes
// from cudaGetSymbolAddress, once per device, in noalloc_scratch() below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoallocMaxDevices];       // device address per device, or null
uint64_t g_noalloc_ctx[kNoallocMaxDevices];     // context the address belongs to

// Device address of the scratch array on `dev` (which must be current).  It
// is looked up once per device and context (a cudaDeviceReset makes a new
// context, in which the array has a new address).
gemm_status_t noalloc_scratch(int dev, unsigned char** out) {
    if (dev < 0 || dev >= kNoallocMaxDevices) return GEMM_ERR_UNSUPPORTED_DEVICE;
    const uint64_t ctx = current_ctx_id(dev);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev] || (ctx && g_noalloc_ctx[dev] != ctx)) {
        void* p = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess) {
            note_cuda_error(e, "cudaGetSymbolAddress(no-alloc scratch)");
            return GEMM_ERR_CUDA;
        }
        g_noalloc_addr[dev] = p;
        g_noalloc_ctx[dev] = ctx;
    }
    *out = static_cast<unsigned char*>(g_noalloc_addr[dev]);
    return GEMM_OK;
}

// Current device, its SM count, and the compute-capability check, read
// through device attributes (no library-side caches are filled).
gemm_status_t noalloc_device(int* dev, int* sms) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaGetDevice");
        return GEMM_ERR_CUDA;
    }
    int major = 0, minor = 0;
    if ((e = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, *dev)) != cudaSuccess ||
        (e = cudaDeviceGetAttribute(sms, cudaDevAttrMultiProcessorCount, *dev)) != cudaSuccess) {
        note_cuda_error(e, "cudaDeviceGetAttribute");
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED_DEVICE;
    return GEMM_OK;
}

// Point a split-K plan at the static scratch: checks the plan's size against
// the maximum and clears the counters it needs on `stream`.
gemm_status_t noalloc_bind_scratch(int dev, const Plan& p, cudaStream_t stream, float** ws,
                                   uint32_t** counters) {
    const size_t counter_bytes = p.n_counters * sizeof(uint32_t);
    const size_t ws_bytes = p.ws_floats * sizeof(float);
    if (counter_bytes > kNoallocCounterBytes ||
        ws_bytes > kNoallocScratchBytes - kNoallocCounterBytes) {
        snprintf(t_last_error, sizeof(t_last_error),
                 "split-K scratch of %zu bytes (+%zu counter bytes) exceeds the "
                 "no-alloc maximum of %zu (+%zu); use fewer K slices or gemm_ex",
                 ws_bytes, counter_bytes, kNoallocScratchBytes - kNoallocCounterBytes,
                 kNoallocCounterBytes);
        return GEMM_ERR_INVALID_VALUE;
    }
    unsigned char* base = nullptr;
    gemm_status_t st = noalloc_scratch(dev, &base);
    if (st != GEMM_OK) return st;
    *counters = reinterpret_cast<uint32_t*>(base);
    *ws = reinterpret_cast<float*>(base + kNoallocCounterBytes);
    // The kernels leave their counters at zero, but a call that gave up a
    // wait may not have; start every call from zero.
    cudaError_t e = cudaMemsetAsync(*counters, 0, counter_bytes, stream);
    if (e != cudaSuccess) {
        note_cuda_error(e, "cudaMemsetAsync(no-alloc counters)");
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // namespace

extern "C" gemm_status_t gemm_ex_noalloc(const void* A, const void* B, void* C, int64_t M,
                                         int64_t N, int64_t K, int64_t lda, int64_t ldb,
                                         int64_t ldc, const gemm_options_t* options,
                                         gemm_stream_t stream_handle) {
    if (!options) return GEMM_ERR_INVALID_VALUE;
    const int dtype = options->dtype;
    if (dtype < 0 || dtype > 5) return GEMM_ERR_INVALID_VALUE;
    gemm_status_t st = check_args(A, B, C, M, N, K, lda, ldb, ldc, dtype_bytes(dtype),
                                  options->trans_a, options->trans_b, options->c_dtype);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev = 0, sms = 0;
    st = noalloc_device(&dev, &sms);
    if (st != GEMM_OK) return st;
    Plan p;
    st = make_plan(dtype, A, B, C, M, N, K, lda, ldb, ldc, *options, sms, &p);
    if (st != GEMM_OK) return st;
    const bool planner_sk = (p.kind == Kind::Sgemm && p.sg.parts[0].sk_mode) ||
                            (p.kind == Kind::Tc && p.tc.sk_mode);
    if (planner_sk && options->stream_k == 0 &&
        p.ws_floats * sizeof(float) > kNoallocScratchBytes - kNoallocCounterBytes) {
        // the planner's own stream-K SGEMM or tail split needs more scratch
        // than the array holds: plan it without (split-K waves or whole tiles)
        gemm_options_t o2 = *options;
        o2.stream_k = 1;
        st = make_plan(dtype, A, B, C, M, N, K, lda, ldb, ldc, o2, sms, &p);
        if (st != GEMM_OK) return st;
    }
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    switch (p.kind) {
        case Kind::Nothing: return GEMM_OK;
        case Kind::ZeroFill:   // the empty sum: beta * C, or zeros
            return launch_status(fill_scale_launch(C, p.ct, M, N, ldc, p.ab == 2 ? p.beta : 0.0f, stream),
                                 "fill_scale");
        case Kind::Generic:
            return launch_status(generic_launch(dtype, A, B, C, p.ct, M, N, K, lda, ldb, ldc, p.ab, p.alpha,
                                                p.beta, p.trans_a, p.trans_b, stream),
                                 "generic_gemm");
        case Kind::Sgemm:
            if (p.ws_floats) {
                st = noalloc_bind_scratch(dev, p, stream, &p.sg.ws, &p.sg.counters);
                if (st != GEMM_OK) return st;
            }
            return launch_status(sgemm_launch(p.sg, stream), "sgemm");
        case Kind::Tc: {
            EncodeTiledFn enc = encode_fn();
            if (!enc) {
                snprintf(t_last_error, sizeof(t_last_error),
                         "cuTensorMapEncodeTiled entry point unavailable");
                return GEMM_ERR_CUDA;
            }
            if (p.ws_floats) {
                st = noalloc_bind_scratch(dev, p, stream, &p.tc.ws, &p.tc.counters);
                if (st != GEMM_OK) return st;
            }
            return launch_status(tc_gemm_launch(p.tc, enc, stream), "tc_gemm");
        }
    }
    return GEMM_ERR_INVALID_VALUE;
}

// ---- host-buffer entry point -------------------------------------------------------
//
// gemm_ex_host: A, B and C in host memory.  C is cut into blocks of row
// panels (of A) by column panels (of B).  The copies in (A panels; B panels
// while the first row panel is being computed), the products (the caller's
// stream) and the copies out (C blocks) run on three streams, so the first C
// block starts back after only a quarter of A and of B have arrived and the
// two copy directions overlap each other and the products.  Device staging
// buffers (B whole, two A row panels, two C row panels), the two copy
// streams and the events belong to the library, one set per (device, caller
// stream), allocated on first use and grown as needed.

namespace {

struct HostPipe {
    uint64_t ctx = 0;   // context the streams, events and buffers belong to
    cudaStream_t s_in = nullptr, s_out = nullptr;
    cudaEvent_t e_start = nullptr, e_a = nullptr, e_b = nullptr, e_blk = nullptr;
    cudaEvent_t e_rowcomp[2] = {}, e_rowout[2] = {};
    void* dB = nullptr;
    size_t dB_bytes = 0;
    void* dA[2] = {};
    size_t dA_bytes = 0;
    void* dC[2] = {};
    size_t dC_bytes = 0;
};

std::mutex g_hp_mu;
std::map<std::pair<int, cudaStream_t>, HostPipe> g_hp;

gemm_status_t grow(void** p, size_t* have, size_t want, const char* what) {
    if (*have >= want) return GEMM_OK;
    if (*p) {
        cudaFree(*p);
        *p = nullptr;
        *have = 0;
    }
    cudaError_t e = cudaMalloc(p, want);
    if (e != cudaSuccess) {
        note_cuda_error(e, what);
        *p = nullptr;
        return GEMM_ERR_OUT_OF_MEMORY;
    }
    ++g_allocs;
    *have = want;
    return GEMM_OK;
}

gemm_status_t host_pipe(int dev, cudaStream_t stream, size_t b_bytes, size_t a_bytes,
                        size_t c_bytes, HostPipe** out) {
    HostPipe& h = g_hp[{dev, stream}];
    const uint64_t ctx = current_ctx_id(dev);
    if (ctx && h.ctx != ctx) {   // made in a context that no longer exists (or none yet)
        h = HostPipe{};
        h.ctx = ctx;
    }
    cudaError_t e = cudaSuccess;
    if (!h.s_in) {
        cudaEvent_t* evs[] = {&h.e_start, &h.e_a, &h.e_b, &h.e_blk, &h.e_rowcomp[0],
                              &h.e_rowcomp[1], &h.e_rowout[0], &h.e_rowout[1]};
        if ((e = cudaStreamCreateWithFlags(&h.s_in, cudaStreamNonBlocking)) != cudaSuccess ||
            (e = cudaStreamCreateWithFlags(&h.s_out, cudaStreamNonBlocking)) != cudaSuccess) {
            note_cuda_error(e, "host pipeline streams");
            return GEMM_ERR_CUDA;
        }
        for (cudaEvent_t* ev : evs) {
            if ((e = cudaEventCreateWithFlags(ev, cudaEventDisableTiming)) != cudaSuccess) {
                note_cuda_error(e, "host pipeline events");
                return GEMM_ERR_CUDA;
            }
        }
    }
    if (h.dB_bytes < b_bytes || h.dA_bytes < a_bytes || h.dC_bytes < c_bytes) {
        // buffers may still be in use by an earlier call on this stream
        if ((e = cudaStreamSynchronize(stream)) != cudaSuccess) {
            note_cuda_error(e, "cudaStreamSynchronize");
            return GEMM_ERR_CUDA;
        }
    }
    gemm_status_t st;
    if ((st = grow(&h.dB, &h.dB_bytes, b_bytes, "cudaMalloc(host pipeline B)")) != GEMM_OK) return st;
    for (int i = 0; i < 2; ++i) {
        // both panel buffers of an operand always have the same size
        size_t ha = h.dA_bytes, hc = h.dC_bytes;
        if ((st = grow(&h.dA[i], &ha, a_bytes, "cudaMalloc(host pipeline A)")) != GEMM_OK) return st;
        if ((st = grow(&h.dC[i], &hc, c_bytes, "cudaMalloc(host pipeline C)")) != GEMM_OK) return st;
    }
    h.dA_bytes = std::max(h.dA_bytes, a_bytes);
    h.dC_bytes = std::max(h.dC_bytes, c_bytes);
    *out = &h;
    return GEMM_OK;
}

// Panel extent along one dimension: a quarter, rounded up to 256, at least
// 512; extents up to 1024 stay whole.
int64_t panel_extent(int64_t n) {
    if (n <= 1024) return n;
    int64_t e = ceil_div(ceil_div(n, 4), 256) * 256;
    return e < 512 ? 512 : e;
}

}  // namespace

extern "C" gemm_status_t gemm_ex_host(const void* A, const void* B, void* C, int64_t M, int64_t N,
                                      int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                                      const gemm_options_t* options, gemm_stream_t stream_handle) {
    if (!options) return GEMM_ERR_INVALID_VALUE;
    const int dtype = options->dtype;
    if (dtype < 0 || dtype > 5) return GEMM_ERR_INVALID_VALUE;
    const size_t es = dtype_bytes(dtype);
    const int ta = options->trans_a, tb = options->trans_b;
    gemm_status_t st = check_args(A, B, C, M, N, K, lda, ldb, ldc, static_cast<int>(es), ta, tb,
                                  options->c_dtype);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) return GEMM_OK;
    int dev;
    DeviceInfo info;
    st = current_device(&dev, &info);
    if (st != GEMM_OK) return st;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);

    const int64_t prow = panel_extent(M), pcol = panel_extent(N);
    const int64_t nrow = ceil_div(M, prow), ncol = ceil_div(N, pcol);
    // Device copies keep the host layout (A row panels, B column panels, each
    // stored as the caller stores the matrix), with row strides rounded up to
    // 16 elements so that every panel is TMA-legal whatever K and N are:
    //   A panel: rows x K (ld ald), or stored transposed K x rows (ld ald);
    //   B: K x N (ld bld), or stored transposed N x K (ld bld);
    //   C panel: rows x N (ld cld).
    auto up16 = [](int64_t x) { return std::max<int64_t>(ceil_div(x, 16) * 16, 16); };
    const int64_t Kp = std::max<int64_t>(K, 1);
    const int64_t ald = ta ? up16(prow) : up16(K);
    const int64_t bld = tb ? up16(K) : up16(N);
    const int64_t cld = up16(N);
    const size_t a_bytes = static_cast<size_t>((ta ? Kp : prow) * ald) * es;
    const size_t b_bytes = static_cast<size_t>((tb ? N : Kp) * bld) * es;
    const size_t ces = static_cast<size_t>(c_elem_bytes(options->c_dtype));
    const size_t c_bytes = static_cast<size_t>(prow * cld) * ces;

    std::lock_guard<std::mutex> lk(g_hp_mu);
    HostPipe* h = nullptr;
    st = host_pipe(dev, stream, b_bytes, a_bytes, c_bytes, &h);
    if (st != GEMM_OK) return st;

    cudaError_t e = cudaSuccess;
#define HP_CHECK(call, what)              \
    do {                                  \
        if ((e = (call)) != cudaSuccess) { \
            note_cuda_error(e, what);     \
            return GEMM_ERR_CUDA;         \
        }                                 \
    } while (0)

    // everything earlier on `stream` (including a previous call's use of the
    // staging buffers) happens before this call's copies
    HP_CHECK(cudaEventRecord(h->e_start, stream), "cudaEventRecord");
    HP_CHECK(cudaStreamWaitEvent(h->s_in, h->e_start, 0), "cudaStreamWaitEvent");
    HP_CHECK(cudaStreamWaitEvent(h->s_out, h->e_start, 0), "cudaStreamWaitEvent");
    // A panel i into buffer i % 2, once row panel i - 2 no longer reads it;
    // `stream` waits for the copy before its next product.
    auto copy_a = [&](int64_t i) -> gemm_status_t {
        const int buf = static_cast<int>(i & 1);
        const int64_t r0 = i * prow;
        const int64_t rows = std::min<int64_t>(prow, M - r0);
        if (i >= 2) HP_CHECK(cudaStreamWaitEvent(h->s_in, h->e_rowcomp[buf], 0), "cudaStreamWaitEvent");
        if (K > 0 && !ta)
            HP_CHECK(cudaMemcpy2DAsync(h->dA[buf], ald * es, static_cast<const char*>(A) + r0 * lda * es,
                                       lda * es, K * es, rows, cudaMemcpyHostToDevice, h->s_in),
                     "cudaMemcpy2DAsync(A panel)");
        if (K > 0 && ta)   // columns r0.. of the stored K x M matrix
            HP_CHECK(cudaMemcpy2DAsync(h->dA[buf], ald * es, static_cast<const char*>(A) + r0 * es,
                                       lda * es, rows * es, K, cudaMemcpyHostToDevice, h->s_in),
                     "cudaMemcpy2DAsync(A panel)");
        HP_CHECK(cudaEventRecord(h->e_a, h->s_in), "cudaEventRecord");
        HP_CHECK(cudaStreamWaitEvent(stream, h->e_a, 0), "cudaStreamWaitEvent");
        // C panel buffer i % 2 is free once row panel i - 2 has been copied out
        if (i >= 2) HP_CHECK(cudaStreamWaitEvent(stream, h->e_rowout[buf], 0), "cudaStreamWaitEvent");
        return GEMM_OK;
    };
    // B column panel j, copied once; `stream` waits for it before its next product
    auto copy_b = [&](int64_t j) -> gemm_status_t {
        if (K == 0) return GEMM_OK;
        const int64_t c0 = j * pcol;
        const int64_t cols = std::min<int64_t>(pcol, N - c0);
        if (!tb)
            HP_CHECK(cudaMemcpy2DAsync(static_cast<char*>(h->dB) + c0 * es, bld * es,
                                       static_cast<const char*>(B) + c0 * es, ldb * es, cols * es, K,
                                       cudaMemcpyHostToDevice, h->s_in),
                     "cudaMemcpy2DAsync(B panel)");
        else   // rows c0.. of the stored N x K matrix
            HP_CHECK(cudaMemcpy2DAsync(static_cast<char*>(h->dB) + c0 * bld * es, bld * es,
                                       static_cast<const char*>(B) + c0 * ldb * es, ldb * es, K * es, cols,
                                       cudaMemcpyHostToDevice, h->s_in),
                     "cudaMemcpy2DAsync(B panel)");
        HP_CHECK(cudaEventRecord(h->e_b, h->s_in), "cudaEventRecord");
        HP_CHECK(cudaStreamWaitEvent(stream, h->e_b, 0), "cudaStreamWaitEvent");
        return GEMM_OK;
    };
    // block (i, j): C's old values in (beta != 0), the product on `stream`,
    // the result out on s_out as soon as it is done
    auto block = [&](int64_t i, int64_t j) -> gemm_status_t {
        const int buf = static_cast<int>(i & 1);
        const int64_t r0 = i * prow, c0 = j * pcol;
        const int64_t rows = std::min<int64_t>(prow, M - r0);
        const int64_t cols = std::min<int64_t>(pcol, N - c0);
        char* cblk = static_cast<char*>(h->dC[buf]) + c0 * ces;
        char* chost = static_cast<char*>(C) + (r0 * ldc + c0) * ces;
        if (options->epilogue && options->beta != 0.0f)   // C's old values take part
            HP_CHECK(cudaMemcpy2DAsync(cblk, cld * ces, chost, ldc * ces, cols * ces, rows,
                                       cudaMemcpyHostToDevice, stream),
                     "cudaMemcpy2DAsync(C block in)");
        const char* bblk = static_cast<const char*>(h->dB) + (tb ? c0 * bld : c0) * es;
        gemm_status_t bst = run(dtype, h->dA[buf], bblk, cblk, rows, cols, K, ald, bld, cld,
                                *options, stream);
        if (bst != GEMM_OK) return bst;
        HP_CHECK(cudaEventRecord(h->e_blk, stream), "cudaEventRecord");
        HP_CHECK(cudaStreamWaitEvent(h->s_out, h->e_blk, 0), "cudaStreamWaitEvent");
        HP_CHECK(cudaMemcpy2DAsync(chost, ldc * ces, cblk, cld * ces, cols * ces, rows,
                                   cudaMemcpyDeviceToHost, h->s_out),
                 "cudaMemcpy2DAsync(C block)");
        return GEMM_OK;
    };
    auto row_done = [&](int64_t i) -> gemm_status_t {
        const int buf = static_cast<int>(i & 1);
        HP_CHECK(cudaEventRecord(h->e_rowcomp[buf], stream), "cudaEventRecord");
        HP_CHECK(cudaEventRecord(h->e_rowout[buf], h->s_out), "cudaEventRecord");
        return GEMM_OK;
    };
#define HP_TRY(call)                      \
    do {                                  \
        gemm_status_t s_ = (call);        \
        if (s_ != GEMM_OK) return s_;     \
    } while (0)

    // Row panels 0 and 1 are multiplied together while B streams in: the
    // copies go A0, B0, A1, B1, B2, ... so the first results -- and the
    // device-to-host copies, the larger half of the traffic -- start after
    // two panels instead of after A0 and all of B.
    const int64_t first = std::min<int64_t>(nrow, 2);
    HP_TRY(copy_a(0));
    for (int64_t j = 0; j < ncol; ++j) {
        HP_TRY(copy_b(j));
        if (j == 0 && first > 1) {
            HP_TRY(block(0, 0));
            HP_TRY(copy_a(1));
            HP_TRY(block(1, 0));
            continue;
        }
        for (int64_t i = 0; i < first; ++i) HP_TRY(block(i, j));
    }
    for (int64_t i = 0; i < first; ++i) HP_TRY(row_done(i));
    // the remaining row panels, one after another, B resident
    for (int64_t i = 2; i < nrow; ++i) {
        HP_TRY(copy_a(i));
        for (int64_t j = 0; j < ncol; ++j) HP_TRY(block(i, j));
        HP_TRY(row_done(i));
    }
#undef HP_TRY
    // later work on `stream` (and the caller's synchronisation) sees all of C
    HP_CHECK(cudaStreamWaitEvent(stream, h->e_rowout[(nrow - 1) & 1], 0), "cudaStreamWaitEvent");
#undef HP_CHECK
    return GEMM_OK;
}
