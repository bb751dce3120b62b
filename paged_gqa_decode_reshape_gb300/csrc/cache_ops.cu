// cache_ops.cu -- KV-cache write path (sm_103a): ReshapeAndCache, Quest
// metadata update / rebuild, and the input checker.
//
// ReshapeAndCache ("Ascend Kernel-to-Serving Pipeline", section
// "ReshapeAndCache"): token t's K and V rows go to block slot / BS, offset
// slot % BS; negative slots are skipped. In the [NB][BS][Hkv][D] layout the
// destination of one token is one contiguous Hkv*D row, so the kernel is a
// 16-byte vectorised row copy, one CTA per token.
//
// Quest metadata: per physical block and KV head, elementwise min/max of K
// over the block's tokens, compared in IEEE totalOrder (-0 < +0) so the result
// is a unique bit pattern whatever the order of the tokens. The fused write
// path does both in one launch.
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

// ------------------------------------------------------------ ReshapeAndCache

__global__ void __launch_bounds__(128) reshape_and_cache_kernel(
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, uint4 *__restrict__ kc,
    uint4 *__restrict__ vc, const int64_t *__restrict__ slots, int row_vecs, int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.x;
    const int64_t slot = __ldg(slots + t);
    if (slot < 0 || slot >= NB * BS) return;  // padding token, or outside the pool
    const int64_t block_idx = slot / BS, block_offset = slot % BS;
    const int64_t dst = (block_idx * BS + block_offset) * row_vecs;
    const int64_t src = t * row_vecs;
    for (int e = threadIdx.x; e < row_vecs; e += blockDim.x) {
        kc[dst + e] = __ldg(key + src + e);
        vc[dst + e] = __ldg(value + src + e);
    }
}

// ---------------------------------------------------------- metadata update

__device__ __forceinline__ uint32_t min_key(uint32_t a, uint32_t b) {
    return bf16_order_key(b) < bf16_order_key(a) ? b : a;
}
__device__ __forceinline__ uint32_t max_key(uint32_t a, uint32_t b) {
    return bf16_order_key(b) > bf16_order_key(a) ? b : a;
}

// Elementwise min/max of 8 packed bf16 values (uint4) in totalOrder.
__device__ __forceinline__ void minmax8(uint4 &lo, uint4 &hi, const uint4 &v) {
    uint32_t *l = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *h = reinterpret_cast<uint32_t *>(&hi);
    const uint32_t *x = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t xl = x[i] & 0xffffu, xh = x[i] >> 16;
        const uint32_t ll = min_key(l[i] & 0xffffu, xl), lh = min_key(l[i] >> 16, xh);
        const uint32_t hl = max_key(h[i] & 0xffffu, xl), hh = max_key(h[i] >> 16, xh);
        l[i] = ll | (lh << 16);
        h[i] = hl | (hh << 16);
    }
}

// Metadata update for token t, run by one warp. The warp of the
// lowest-index token landing in a physical block (its "leader") gathers every
// token of the call in that block and writes the block's new metadata; the
// other warps do nothing. So each block is written by exactly one warp and no
// atomics are needed. The slot scan is one coalesced pass (ballots over 32
// tokens at a time); in a decode step a block receives one token, so the
// leader has no further members to visit.
__device__ __forceinline__ void meta_update_warp(uint4 *__restrict__ kmin, uint4 *__restrict__ kmax,
                                                 const uint4 *__restrict__ key,
                                                 const int64_t *__restrict__ slots, int64_t T,
                                                 int64_t t, int64_t s, int row_vecs, int BS,
                                                 int64_t NB, int lane) {
    const int64_t p = s / BS;
    bool reset = (s % BS) == 0;
    int64_t first_member_chunk = -1;   // first 32-token chunk holding a later token of block p
    for (int64_t u0 = 0; u0 < T; u0 += 32) {
        const int64_t u = u0 + lane;
        const int64_t su = u < T ? __ldg(slots + u) : -1;
        const bool in_blk = su >= 0 && su < NB * BS && su / BS == p;
        if (__any_sync(0xffffffffu, in_blk && u < t)) return;  // not the leader
        const unsigned later = __ballot_sync(0xffffffffu, in_blk && u > t);
        reset |= __any_sync(0xffffffffu, in_blk && u > t && (su % BS) == 0);
        if (later && first_member_chunk < 0) first_member_chunk = u0;
    }
    // leader: start from the old metadata or, if the block starts fresh, from
    // this token; then merge every later token of the call in the block
    for (int e = lane; e < row_vecs; e += 32) {
        const uint4 kt = __ldg(key + t * row_vecs + e);
        uint4 lo = kt, hi = kt;
        if (!reset) {
            lo = kmin[p * row_vecs + e];
            hi = kmax[p * row_vecs + e];
            minmax8(lo, hi, kt);
        }
        kmin[p * row_vecs + e] = lo;
        kmax[p * row_vecs + e] = hi;
    }
    if (first_member_chunk < 0) return;
    for (int64_t u0 = first_member_chunk; u0 < T; u0 += 32) {
        const int64_t u = u0 + lane;
        const int64_t su = u < T ? __ldg(slots + u) : -1;
        unsigned m = __ballot_sync(0xffffffffu, su >= 0 && su < NB * BS && su / BS == p && u > t);
        while (m) {
            const int bit = __ffs(m) - 1;
            m &= m - 1;
            const int64_t tu = u0 + bit;
            for (int e = lane; e < row_vecs; e += 32) {
                uint4 lo = kmin[p * row_vecs + e], hi = kmax[p * row_vecs + e];
                minmax8(lo, hi, __ldg(key + tu * row_vecs + e));
                kmin[p * row_vecs + e] = lo;
                kmax[p * row_vecs + e] = hi;
            }
        }
    }
}

// quest_update_meta: one warp per token.
__global__ void __launch_bounds__(256) update_meta_kernel(
    uint4 *__restrict__ kmin, uint4 *__restrict__ kmax, const uint4 *__restrict__ key,
    const int64_t *__restrict__ slots, int64_t T, int row_vecs, int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int64_t s = __ldg(slots + t);
    if (s < 0 || s >= NB * BS) return;
    meta_update_warp(kmin, kmax, key, slots, T, t, s, row_vecs, BS, NB, lane);
}

// The write path in one pass (ReshapeAndCache followed by the metadata
// update): one warp per token copies its K and V rows into the cache, then
// takes part in the metadata update of its block.
__global__ void __launch_bounds__(256) write_quest_kernel(
    uint4 *__restrict__ kc, uint4 *__restrict__ vc, uint4 *__restrict__ kmin,
    uint4 *__restrict__ kmax, const uint4 *__restrict__ key, const uint4 *__restrict__ value,
    const int64_t *__restrict__ slots, int64_t T, int row_vecs, int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int64_t s = __ldg(slots + t);
    // the token's K and V rows do not depend on its slot: load the first two
    // vectors per lane while the slot is in flight
    const int64_t src = t * row_vecs;
    const uint4 zero = make_uint4(0, 0, 0, 0);
    const uint4 k0 = lane < row_vecs ? __ldg(key + src + lane) : zero;
    const uint4 v0 = lane < row_vecs ? __ldg(value + src + lane) : zero;
    const uint4 k1 = lane + 32 < row_vecs ? __ldg(key + src + lane + 32) : zero;
    const uint4 v1 = lane + 32 < row_vecs ? __ldg(value + src + lane + 32) : zero;
    if (s < 0 || s >= NB * BS) return;  // padding token, or outside the pool
    const int64_t dst = s * row_vecs;   // (block * BS + offset) rows of Hkv*D
    for (int e = lane; e < row_vecs; e += 32) {
        kc[dst + e] = e < 32 ? k0 : (e < 64 ? k1 : __ldg(key + src + e));
        vc[dst + e] = e < 32 ? v0 : (e < 64 ? v1 : __ldg(value + src + e));
    }
    meta_update_warp(kmin, kmax, key, slots, T, t, s, row_vecs, BS, NB, lane);
}

// ---------------------------------------------------------- metadata rebuild

// One CTA per (logical block j, sequence b): min/max over the block's valid
// tokens, read straight from the cache.
__global__ void __launch_bounds__(64) rebuild_meta_kernel(
    uint4 *__restrict__ kmin, uint4 *__restrict__ kmax, const uint4 *__restrict__ kc,
    const int32_t *__restrict__ bt, int MBS, const int32_t *__restrict__ ctx, int row_vecs,
    int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int j = blockIdx.x, b = blockIdx.y;
    const int c = min(max(__ldg(ctx + b), 0), MBS * BS);
    if (j * BS >= c) return;
    const int p = __ldg(bt + int64_t(b) * MBS + j);
    if (p < 0 || int64_t(p) >= NB) return;
    const int nv = min(BS, c - j * BS);
    for (int e = threadIdx.x; e < row_vecs; e += blockDim.x) {
        uint4 lo = __ldg(kc + (int64_t(p) * BS) * row_vecs + e), hi = lo;
        for (int o = 1; o < nv; ++o) minmax8(lo, hi, __ldg(kc + (int64_t(p) * BS + o) * row_vecs + e));
        kmin[int64_t(p) * row_vecs + e] = lo;
        kmax[int64_t(p) * row_vecs + e] = hi;
    }
}

// ------------------------------------------------------------- input checker

__global__ void __launch_bounds__(256) check_metadata_kernel(
    int32_t *counts, const int64_t *__restrict__ slots, int64_t T, const int32_t *__restrict__ bt,
    int MBS, const int32_t *__restrict__ ctx, int B, int BS, int64_t NB) {
    const int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x;
    if (slots && i < T) {
        const int64_t s = slots[i];
        if (s >= NB * BS) atomicAdd(counts + 0, 1);
        if (s >= 0) {
            for (int64_t u = 0; u < i; ++u)
                if (slots[u] == s) {
                    atomicAdd(counts + 3, 1);
                    break;
                }
        }
    }
    if (ctx && i < B) {
        const int c = ctx[i];
        if (c < 0 || int64_t(c) > int64_t(MBS) * BS) atomicAdd(counts + 1, 1);
        if (bt) {
            const int cc = min(max(c, 0), MBS * BS);
            const int nblk = (cc + BS - 1) / BS;
            int bad = 0;
            for (int j = 0; j < nblk; ++j) {
                const int p = bt[i * MBS + j];
                bad += (p < 0 || int64_t(p) >= NB);
            }
            if (bad) atomicAdd(counts + 2, bad);
        }
    }
}

}  // namespace

cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *kc,
                                     uint16_t *vc, const int64_t *slots, int64_t T, int Hkv, int D,
                                     int BS, int64_t NB, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int row_vecs = Hkv * D / 8;
    return launch_pdl(reshape_and_cache_kernel, dim3(unsigned(T)), dim3(128), 0, stream,
                      reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value),
                      reinterpret_cast<uint4 *>(kc), reinterpret_cast<uint4 *>(vc), slots, row_vecs,
                      BS, NB);
}

cudaError_t launch_update_meta(uint16_t *kmin, uint16_t *kmax, const uint16_t *key,
                               const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                               cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int row_vecs = Hkv * D / 8;
    const int warps = 8;
    const unsigned grid = unsigned((T + warps - 1) / warps);
    return launch_pdl(update_meta_kernel, dim3(grid), dim3(warps * 32), 0, stream,
                      reinterpret_cast<uint4 *>(kmin), reinterpret_cast<uint4 *>(kmax),
                      reinterpret_cast<const uint4 *>(key), slots, T, row_vecs, BS, NB);
}

cudaError_t launch_write_quest(uint16_t *kc, uint16_t *vc, uint16_t *kmin, uint16_t *kmax,
                               const uint16_t *key, const uint16_t *value, const int64_t *slots,
                               int64_t T, int Hkv, int D, int BS, int64_t NB, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int row_vecs = Hkv * D / 8;
    const int warps = 8;
    const unsigned grid = unsigned((T + warps - 1) / warps);
    return launch_pdl(write_quest_kernel, dim3(grid), dim3(warps * 32), 0, stream,
                      reinterpret_cast<uint4 *>(kc), reinterpret_cast<uint4 *>(vc),
                      reinterpret_cast<uint4 *>(kmin), reinterpret_cast<uint4 *>(kmax),
                      reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value),
                      slots, T, row_vecs, BS, NB);
}

cudaError_t launch_rebuild_meta(uint16_t *kmin, uint16_t *kmax, const uint16_t *kc,
                                const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hkv,
                                int D, int BS, int64_t NB, cudaStream_t stream) {
    const int row_vecs = Hkv * D / 8;
    const dim3 grid{unsigned(MBS), unsigned(B), 1u};
    return launch_pdl(rebuild_meta_kernel, grid, dim3(64), 0, stream,
                      reinterpret_cast<uint4 *>(kmin), reinterpret_cast<uint4 *>(kmax),
                      reinterpret_cast<const uint4 *>(kc), bt, MBS, ctx, row_vecs, BS, NB);
}

cudaError_t launch_check_metadata(int32_t *counts, const int64_t *slots, int64_t T,
                                  const int32_t *bt, int MBS, const int32_t *ctx, int B, int BS,
                                  int64_t NB, cudaStream_t stream) {
    cudaError_t e = cudaMemsetAsync(counts, 0, 4 * sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
    const int64_t n = T > B ? T : B;
    if (n == 0) return cudaSuccess;
    check_metadata_kernel<<<unsigned((n + 255) / 256), 256, 0, stream>>>(counts, slots, T, bt, MBS,
                                                                          ctx, B, BS, NB);
    return cudaGetLastError();
}

}  // namespace pa
