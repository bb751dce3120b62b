// common.cuh -- device helpers shared by the paged decode kernels (sm_103a).
//
// Inline PTX for the pieces the kernels are built from: mbarriers, TMA tile
// loads (cp.async.bulk.tensor) with 128-byte swizzle, ldmatrix, bf16 mma.sync,
// movmatrix, ex2. Everything here is warp- or thread-level; no kernel state.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <utility>
#include <vector>

namespace pa {

constexpr int kStatusTimeout = 1;  // bit in a workspace status word: a wait gave up

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ----------------------------------------------------------------- mbarrier

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

// Order this thread's earlier shared-memory accesses before later accesses
// of the async (TMA) proxy to the same memory.
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// Order this thread's earlier global-memory writes before later accesses of
// the async (TMA) proxy to the same memory (a kernel that writes cache rows
// and then loads them with TMA).
__device__ __forceinline__ void fence_proxy_async_global() {
    asm volatile("fence.proxy.async.global;" ::: "memory");
}

// Make barrier initialisation visible to the async (TMA) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Atomic add at GPU scope with acquire-release semantics: the caller's earlier
// writes (and those it observed) are published before the add, and later reads
// see what the other adders published before theirs.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int *p, int v) {
    int old;
    asm volatile("atom.acq_rel.gpu.global.add.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

// 1 / x for x a normal power of two 2^k with k <= 126 (the result 2^-k is
// normal too), exact: the exponent field is negated around the bias.
__device__ __forceinline__ float rcp_pow2(float x) { return __int_as_float(0x7f000000 - __float_as_int(x)); }

// Acquire load at GPU scope (a counter other CTAs update with release
// semantics): what those CTAs published before their update is visible to
// this thread's later reads.
__device__ __forceinline__ int ld_acquire_s32(const int *p) {
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream is still
// running; pdl_wait() blocks until that kernel has completed and its memory
// is visible (a no-op for an ordinary launch). pdl_trigger() lets the next
// kernel in the stream launch early.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase with the given parity to complete, for at most
// `limit_ns` nanoseconds. Returns false on timeout (the caller records it).
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_timer_ns() - t0 > limit_ns) return false;
    }
}

// ---------------------------------------------------------------------- TMA

__device__ __forceinline__ uint64_t l2_policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// Hint: bring one 128-byte line into L2 (no value is returned, nothing is
// cached closer to the SM, so a later write by another kernel is still seen).
__device__ __forceinline__ void prefetch_l2(const void *p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_tensormap(const CUtensorMap *map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// 4-D tiled TMA load into shared memory, completion counted on `bar`.
__device__ __forceinline__ void tma_load_4d(uint32_t dst, const CUtensorMap *map, uint32_t bar,
                                            int c0, int c1, int c2, int c3, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        ".L2::cache_hint [%0], [%1, {%3, %4, %5, %6}], [%2], %7;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(bar), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "l"(policy)
        : "memory");
}

// 1-D bulk copy of `bytes` contiguous bytes (16-byte aligned, multiple of 16)
// into shared memory, completion counted on `bar`.
__device__ __forceinline__ void bulk_load_1d(uint32_t dst, const void *src, uint32_t bytes, uint32_t bar,
                                             uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1], %2, [%3], %4;" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(bar), "l"(policy)
        : "memory");
}

// ------------------------------------------------------------ tensor cores

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t addr, uint32_t &r0, uint32_t &r1,
                                              uint32_t &r2, uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr)
                 : "memory");
}

// D = A * B + D, m16n8k16, bf16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_bf16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D = A * B + D, m16n8k16, f16 inputs, fp32 accumulators.
__device__ __forceinline__ void mma_f16(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                        uint32_t a3, uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// Transpose one 8x8 b16 tile held as an m8n8 fragment across the warp.
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
    uint32_t y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
    return y;
}

// 2^x (hardware approximation; ex2(-inf) = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float y;
    asm volatile("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint32_t pack_f16x2(float lo, float hi) {
    __half2 v = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}
__device__ __forceinline__ float f16_lo(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v & 0xffffu)));
}
__device__ __forceinline__ float f16_hi(uint32_t v) {
    return __half2float(__ushort_as_half(static_cast<unsigned short>(v >> 16)));
}

// An f16 pair times r (rounded to f16), each product rounded to nearest.
__device__ __forceinline__ uint32_t scale_f16x2(uint32_t v, float r) {
    const __half2 m = __hmul2(*reinterpret_cast<const __half2 *>(&v), __float2half2_rn(r));
    return *reinterpret_cast<const uint32_t *>(&m);
}

// Two E4M3 codes (low byte first) to an f16 pair (low half first); exact.
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t two_codes) {
    const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(
        static_cast<__nv_fp8x2_storage_t>(two_codes & 0xffffu), __NV_E4M3);
    return uint32_t(h.x) | (uint32_t(h.y) << 16);
}

// Four E4M3 codes (bytes 0..3) to two f16 pairs: lo = bytes 0, 1 and hi =
// bytes 2, 3, each with the lower byte in the lower half; exact.
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t four, uint32_t &lo, uint32_t &hi) {
    asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, l;\n\tcvt.rn.f16x2.e4m3x2 %1, h;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(four));
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

// IEEE totalOrder key of a bf16 bit pattern (numeric order, -0 < +0).
__device__ __forceinline__ uint32_t bf16_order_key(uint32_t h) {
    return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}

// Elementwise min / max (totalOrder) of two packed bf16 values with x.
__device__ __forceinline__ void minmax_bf16x2(uint32_t &lo, uint32_t &hi, uint32_t x) {
    uint32_t l = 0, h = 0;
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        const uint32_t xv = (x >> (16 * i)) & 0xffffu;
        const uint32_t lv = (lo >> (16 * i)) & 0xffffu, hv = (hi >> (16 * i)) & 0xffffu;
        l |= (bf16_order_key(xv) < bf16_order_key(lv) ? xv : lv) << (16 * i);
        h |= (bf16_order_key(xv) > bf16_order_key(hv) ? xv : hv) << (16 * i);
    }
    lo = l;
    hi = h;
}

// IEEE totalOrder key of an fp32 value.
__device__ __forceinline__ uint32_t f32_order_key(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// keys[j] = totalOrder key of row[j] for j < n, by all THREADS threads of a
// CTA: each thread issues U independent loads before storing any, so a row
// costs a few L2 round trips rather than one per element a thread holds.
template <int THREADS, int U = 16>
__device__ __forceinline__ void cta_load_keys(uint32_t *keys, const float *row, int n) {
    for (int j0 = threadIdx.x; j0 < n; j0 += THREADS * U) {
        float v[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * THREADS;
            v[u] = j < n ? __ldcg(row + j) : 0.f;
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int j = j0 + u * THREADS;
            if (j < n) keys[j] = f32_order_key(v[u]);
        }
    }
}

// ---- Top-K of a row of totalOrder keys, by all THREADS threads of a CTA
// (the Quest block selection: the topk largest scores, ties to the lower
// block index). key_of(j) gives key j < n (n > topk).
//
// Threshold: the topk-th largest key `thr`, and `keq`, how many keys equal
// to it are taken (the keq lowest-index ones; every key above thr is taken).
// Radix select from the top in digits of up to 8 bits, starting at the
// highest bit where the row's smallest and largest keys differ (the scores of
// a row share their sign, exponent and often more, so a fixed first digit
// would put every key into one bin and serialise its atomic adds).
// hist: HC * 256 ints of shared memory, HC histogram copies (warp w adds to
// copy w % HC: the keys of a row crowd into few bins, and copies spread the
// atomic adds of different warps over different addresses); red: at least
// 2 * THREADS / 32 + 3 ints. When the bin holding the topk-th key ends
// exactly at the topk-th key, the selection is every key from that bin's
// lowest value up: the passes stop there, with thr one below that value and
// keq = 0 (the same selection as the full descent).
template <int THREADS, int HC = 1, typename KeyOf>
__device__ __forceinline__ void cta_topk_threshold(KeyOf key_of, int n, int topk, int *hist, int *red,
                                                   uint32_t &thr, int &keq) {
    static_assert(HC >= 1 && HC <= THREADS / 32, "one histogram copy per warp at most");
    constexpr int NW = THREADS / 32, U = 4;  // U keys per thread in flight
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t lo = 0xffffffffu, hi = 0u;
    for (int j0 = tid; j0 < n; j0 += U * THREADS) {
        uint32_t u[U];
#pragma unroll
        for (int i = 0; i < U; ++i) {
            const int j = j0 + i * THREADS;
            u[i] = j < n ? key_of(j) : 0u;
        }
#pragma unroll
        for (int i = 0; i < U; ++i)
            if (j0 + i * THREADS < n) {
                lo = min(lo, u[i]);
                hi = max(hi, u[i]);
            }
    }
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) {
        lo = min(lo, __shfl_xor_sync(0xffffffffu, lo, o));
        hi = max(hi, __shfl_xor_sync(0xffffffffu, hi, o));
    }
    if (lane == 0) {
        red[warp] = int(lo);
        red[NW + warp] = int(hi);
    }
    __syncthreads();
    lo = 0xffffffffu;
    hi = 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
        lo = min(lo, uint32_t(red[w]));
        hi = max(hi, uint32_t(red[NW + w]));
    }
    int k = topk;
    if (lo == hi) {  // every key equal: the topk lowest indices
        thr = hi;
        keq = k;
        __syncthreads();  // red may be reused by the caller
        return;
    }
    const int top = 31 - __clz(lo ^ hi);  // the keys agree on every bit above this one
    uint32_t mask = top == 31 ? 0u : ~((2u << top) - 1u);
    uint32_t prefix = hi & mask;
    for (int h = top; h >= 0;) {
        const int l = h >= 7 ? h - 7 : 0;
        const uint32_t dm = (2u << (h - l)) - 1u;  // digit of bits l..h
        for (int i = tid; i < HC * 256; i += THREADS) hist[i] = 0;
        __syncthreads();
        int *my_hist = hist + (warp % HC) * 256;
        for (int j0 = tid; j0 < n; j0 += U * THREADS) {
            uint32_t u[U];
#pragma unroll
            for (int i = 0; i < U; ++i) {
                const int j = j0 + i * THREADS;
                u[i] = j < n ? key_of(j) : 0u;
            }
#pragma unroll
            for (int i = 0; i < U; ++i)
                if (j0 + i * THREADS < n && (u[i] & mask) == prefix) atomicAdd(&my_hist[(u[i] >> l) & dm], 1);
        }
        __syncthreads();
        if (warp == 0) {
            // lane t holds digits 255-8t .. 248-8t (descending)
            int cnt[8], sum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cnt[i] = 0;
#pragma unroll
                for (int c = 0; c < HC; ++c) cnt[i] += hist[c * 256 + 255 - 8 * lane - i];
                sum += cnt[i];
            }
            int incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int before = incl - sum;
            if (before < k && k <= incl) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (before + cnt[i] >= k) {
                        red[2 * NW] = 255 - 8 * lane - i;
                        red[2 * NW + 1] = before;
                        red[2 * NW + 2] = before + cnt[i] == k;
                        break;
                    }
                    before += cnt[i];
                }
            }
        }
        __syncthreads();
        prefix |= uint32_t(red[2 * NW]) << l;
        mask |= dm << l;
        k -= red[2 * NW + 1];
        h = l - 1;
        if (red[2 * NW + 2] && prefix != 0u && h >= 0) {
            // every key of the bin is taken: all keys >= prefix (low bits 0)
            thr = prefix - 1u;
            keq = 0;
            __syncthreads();  // red may be reused by the caller
            return;
        }
    }
    thr = prefix;
    keq = k;
    __syncthreads();  // red may be reused by the caller
}

// The selection for a threshold: every key above thr and the keq lowest-index
// keys equal to it, emitted as emit(r, j) with r the rank of block j among
// the selected (ascending j). The row is cut into one contiguous range per
// thread (ranges ascending with the thread index): each thread counts its
// keys above and equal to thr, an exclusive scan over the CTA gives every
// thread its first rank and the equal keys before it, then each thread emits
// its own range in order. red: at least 2 * THREADS / 32 ints.
template <int THREADS, typename KeyOf, typename Emit>
__device__ __forceinline__ void cta_topk_emit(KeyOf key_of, int n, uint32_t thr, int keq, int *red, Emit emit) {
    constexpr int NW = THREADS / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + THREADS - 1) / THREADS;  // keys per thread
    const int j0 = min(n, tid * per), j1 = min(n, j0 + per);
    int cgt = 0, ceq = 0;
    for (int j = j0; j < j1; ++j) {
        const uint32_t u = key_of(j);
        cgt += u > thr;
        ceq += u == thr;
    }
    // exclusive scans of the two counts over the warp, then over the warps
    int xgt = cgt, xeq = ceq;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int a = __shfl_up_sync(0xffffffffu, xgt, o), b = __shfl_up_sync(0xffffffffu, xeq, o);
        if (lane >= o) {
            xgt += a;
            xeq += b;
        }
    }
    if (lane == 31) {
        red[warp] = xgt;
        red[NW + warp] = xeq;
    }
    xgt -= cgt;
    xeq -= ceq;
    __syncthreads();
    for (int w = 0; w < warp; ++w) {
        xgt += red[w];
        xeq += red[NW + w];
    }
    // rank of the thread's first selected key: the keys above thr before it,
    // plus the equal keys before it that are taken
    int pos = xgt + min(max(keq, 0), xeq), seen_eq = xeq;
    for (int j = j0; j < j1; ++j) {
        const uint32_t u = key_of(j);
        const bool take = u > thr || (u == thr && seen_eq < keq);
        seen_eq += u == thr;
        if (take) emit(pos++, j);
    }
    __syncthreads();  // red may be reused by the caller
}

// Host side: ask once per (device, kernel) for the largest shared-memory
// carveout, the split the decode kernel needs, so that consecutive kernels of
// the library never make the SMs reconfigure between them.
inline void carveout_once(const void *kernel) {
    static std::mutex mu;
    static std::vector<std::pair<int, const void *>> done;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return;
    std::lock_guard<std::mutex> lock(mu);
    for (const auto &d : done)
        if (d.first == dev && d.second == kernel) return;
    cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    done.emplace_back(dev, kernel);
}

// Host side: launch a kernel with programmatic stream serialization allowed.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
    carveout_once(reinterpret_cast<const void *>(kernel));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace pa
