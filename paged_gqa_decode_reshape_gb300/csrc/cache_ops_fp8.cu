// cache_ops_fp8.cu -- write path of an 8-bit (E4M3) KV cache (sm_103a):
// ReshapeAndCache with quantisation, Quest metadata on the stored codes, and
// the metadata rebuild.
//
// Same slot arithmetic as the bf16 path ("Ascend Kernel-to-Serving
// Pipeline", section "ReshapeAndCache": block slot / BS, offset slot % BS,
// negative slots skipped). Element d of KV head h is stored as the E4M3 code
// of fl32(x / scale[h]), rounded to nearest (ties to even) and saturated to
// +-448; a NaN element is stored as 0x7F. Quest metadata of an E4M3 cache is
// the elementwise min / max of the stored codes in numeric order (-0 < +0),
// with the bf16 path's update rule (reset when a token of the call lands at
// offset 0 of the block, else merge).
//
// One warp per token; a lane converts 8 bf16 elements (one 16-byte load) into
// 8 codes (one 8-byte K store; eight V bytes, one per dim row of the V layout).
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

// E4M3 codes of 8 bf16 elements of one KV head, divided by its scale.
__device__ __forceinline__ uint2 quantize8(const uint4 &x, float scale) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&x);
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t v = w[2 * i + j];
            const float a = __fdiv_rn(bf16_lo(v), scale), b = __fdiv_rn(bf16_hi(v), scale);
            uint32_t pair = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
            if (a != a) pair = (pair & 0xff00u) | 0x7fu;  // one NaN code
            if (b != b) pair = (pair & 0x00ffu) | 0x7f00u;
            word |= (pair & 0xffffu) << (16 * j);
        }
        out[i] = word;
    }
    return make_uint2(out[0], out[1]);
}

// numeric order key of an E4M3 code (-0 below +0)
__device__ __forceinline__ uint32_t e4m3_key(uint32_t c) { return (c & 0x80u) ? (~c & 0x7fu) : (c | 0x80u); }

// elementwise min / max of 8 packed codes
__device__ __forceinline__ void minmax8_e4m3(uint2 &lo, uint2 &hi, const uint2 &v) {
    uint32_t *l = reinterpret_cast<uint32_t *>(&lo);
    uint32_t *h = reinterpret_cast<uint32_t *>(&hi);
    const uint32_t *x = reinterpret_cast<const uint32_t *>(&v);
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t nl = 0, nh = 0;
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const uint32_t xb = (x[i] >> (8 * k)) & 0xffu;
            const uint32_t lb = (l[i] >> (8 * k)) & 0xffu, hb = (h[i] >> (8 * k)) & 0xffu;
            nl |= (e4m3_key(xb) < e4m3_key(lb) ? xb : lb) << (8 * k);
            nh |= (e4m3_key(xb) > e4m3_key(hb) ? xb : hb) << (8 * k);
        }
        l[i] = nl;
        h[i] = nh;
    }
}

// Metadata update for token t by its warp: the warp of the lowest-index token
// of the call landing in a physical block gathers every token of the call in
// that block and writes the block's codes' min / max; other warps return.
// Row vectors: row_vecs = Hkv * D / 8, each 8 elements of one KV head.
__device__ __forceinline__ void meta_update_warp_fp8(uint2 *__restrict__ kmin, uint2 *__restrict__ kmax,
                                                     const uint4 *__restrict__ key,
                                                     const float *__restrict__ k_scale,
                                                     const int64_t *__restrict__ slots, int64_t T,
                                                     int64_t t, int64_t s, int row_vecs, int vecs_per_head,
                                                     int BS, int64_t NB, int lane) {
    const int64_t p = s / BS;
    bool reset = (s % BS) == 0;
    int64_t first_member_chunk = -1;
    for (int64_t u0 = 0; u0 < T; u0 += 32) {
        const int64_t u = u0 + lane;
        const int64_t su = u < T ? __ldg(slots + u) : -1;
        const bool in_blk = su >= 0 && su < NB * BS && su / BS == p;
        if (__any_sync(0xffffffffu, in_blk && u < t)) return;  // not the leader
        const unsigned later = __ballot_sync(0xffffffffu, in_blk && u > t);
        reset |= __any_sync(0xffffffffu, in_blk && u > t && (su % BS) == 0);
        if (later && first_member_chunk < 0) first_member_chunk = u0;
    }
    for (int e = lane; e < row_vecs; e += 32) {
        const uint2 kt = quantize8(__ldg(key + t * row_vecs + e), __ldg(k_scale + e / vecs_per_head));
        uint2 lo = kt, hi = kt;
        if (!reset) {
            lo = kmin[p * row_vecs + e];
            hi = kmax[p * row_vecs + e];
            minmax8_e4m3(lo, hi, kt);
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
                uint2 lo = kmin[p * row_vecs + e], hi = kmax[p * row_vecs + e];
                minmax8_e4m3(lo, hi, quantize8(__ldg(key + tu * row_vecs + e),
                                               __ldg(k_scale + e / vecs_per_head)));
                kmin[p * row_vecs + e] = lo;
                kmax[p * row_vecs + e] = hi;
            }
        }
    }
}

// ReshapeAndCache into an E4M3 cache (META: then the metadata update). K
// codes go to the token's row of [NB][BS][Hkv][D]; V codes to the V layout:
// per block and KV head a [D][16] byte matrix, token o at byte
// 4 * ((o % 8) / 2) + 2 * (o / 8) + (o % 2) of each dim's row.
template <bool META>
__global__ void __launch_bounds__(256) write_fp8_kernel(
    uint2 *__restrict__ kc, uint8_t *__restrict__ vc, uint2 *__restrict__ kmin, uint2 *__restrict__ kmax,
    const uint4 *__restrict__ key, const uint4 *__restrict__ value, const float *__restrict__ k_scale,
    const float *__restrict__ v_scale, const int64_t *__restrict__ slots, int64_t T, int row_vecs,
    int vecs_per_head, int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int64_t s = __ldg(slots + t);
    if (s < 0 || s >= NB * BS) return;  // padding token, or outside the pool
    const int64_t dst = s * row_vecs;   // (block * BS + offset) rows of Hkv*D codes
    const int64_t p = s / BS;
    const int o = int(s % BS);
    const int pos = 4 * ((o & 7) >> 1) + 2 * (o >> 3) + (o & 1);
    const int D = vecs_per_head * 8, Hkv = row_vecs / vecs_per_head;
    for (int e = lane; e < row_vecs; e += 32) {
        const int h = e / vecs_per_head, d0 = (e - h * vecs_per_head) * 8;
        kc[dst + e] = quantize8(__ldg(key + t * row_vecs + e), __ldg(k_scale + h));
        const uint2 v = quantize8(__ldg(value + t * row_vecs + e), __ldg(v_scale + h));
        uint8_t *vrow = vc + ((p * Hkv + h) * D + d0) * 16 + pos;
#pragma unroll
        for (int i = 0; i < 8; ++i) vrow[16 * i] = uint8_t(((i < 4 ? v.x : v.y) >> (8 * (i & 3))) & 0xffu);
    }
    if (META)
        meta_update_warp_fp8(kmin, kmax, key, k_scale, slots, T, t, s, row_vecs, vecs_per_head, BS, NB,
                             lane);
}

// the metadata update alone (quest_update_meta_fp8), one warp per token
__global__ void __launch_bounds__(256) update_meta_fp8_kernel(
    uint2 *__restrict__ kmin, uint2 *__restrict__ kmax, const uint4 *__restrict__ key,
    const float *__restrict__ k_scale, const int64_t *__restrict__ slots, int64_t T, int row_vecs,
    int vecs_per_head, int BS, int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int64_t t = int64_t(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int lane = threadIdx.x & 31;
    if (t >= T) return;
    const int64_t s = __ldg(slots + t);
    if (s < 0 || s >= NB * BS) return;
    meta_update_warp_fp8(kmin, kmax, key, k_scale, slots, T, t, s, row_vecs, vecs_per_head, BS, NB, lane);
}

// One CTA per (logical block j, sequence b): min / max of the stored codes
// over the block's valid tokens.
__global__ void __launch_bounds__(64) rebuild_meta_fp8_kernel(
    uint2 *__restrict__ kmin, uint2 *__restrict__ kmax, const uint2 *__restrict__ kc,
    const int32_t *__restrict__ bt, int MBS, const int32_t *__restrict__ ctx, int row_vecs, int BS,
    int64_t NB) {
    pdl_trigger();
    pdl_wait();
    const int j = blockIdx.x, b = blockIdx.y;
    const int c = min(max(__ldg(ctx + b), 0), MBS * BS);
    if (j * BS >= c) return;
    const int p = __ldg(bt + int64_t(b) * MBS + j);
    if (p < 0 || int64_t(p) >= NB) return;
    const int nv = min(BS, c - j * BS);
    for (int e = threadIdx.x; e < row_vecs; e += blockDim.x) {
        uint2 lo = __ldg(kc + (int64_t(p) * BS) * row_vecs + e), hi = lo;
        for (int o = 1; o < nv; ++o)
            minmax8_e4m3(lo, hi, __ldg(kc + (int64_t(p) * BS + o) * row_vecs + e));
        kmin[int64_t(p) * row_vecs + e] = lo;
        kmax[int64_t(p) * row_vecs + e] = hi;
    }
}

}  // namespace

cudaError_t launch_write_fp8(uint8_t *kc, uint8_t *vc, uint8_t *kmin, uint8_t *kmax, const uint16_t *key,
                             const uint16_t *value, const float *k_scale, const float *v_scale,
                             const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                             cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int row_vecs = Hkv * D / 8, vph = D / 8;
    // One warp per CTA, so a decode step's few tokens spread over as many
    // SMs. A token's V bytes touch Hkv * D / 8 separate 128-byte lines (one
    // byte per 16-byte row), and those uncoalesced stores queue in the
    // load/store unit of the SM that issues them: with 8 warps per CTA, 16
    // tokens took 16.0 us on 2 SMs against 11.9 us on 16.
    const int warps = 1;
    const unsigned grid = unsigned((T + warps - 1) / warps);
    auto *kfn = kmin ? write_fp8_kernel<true> : write_fp8_kernel<false>;
    return launch_pdl(kfn, dim3(grid), dim3(warps * 32), 0, stream, reinterpret_cast<uint2 *>(kc), vc,
                      reinterpret_cast<uint2 *>(kmin),
                      reinterpret_cast<uint2 *>(kmax), reinterpret_cast<const uint4 *>(key),
                      reinterpret_cast<const uint4 *>(value), k_scale, v_scale, slots, T, row_vecs, vph,
                      BS, NB);
}

cudaError_t launch_update_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint16_t *key, const float *k_scale,
                                   const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                                   cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int row_vecs = Hkv * D / 8, vph = D / 8;
    const int warps = 8;
    const unsigned grid = unsigned((T + warps - 1) / warps);
    return launch_pdl(update_meta_fp8_kernel, dim3(grid), dim3(warps * 32), 0, stream,
                      reinterpret_cast<uint2 *>(kmin), reinterpret_cast<uint2 *>(kmax),
                      reinterpret_cast<const uint4 *>(key), k_scale, slots, T, row_vecs, vph, BS, NB);
}

cudaError_t launch_rebuild_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint8_t *kc, const int32_t *bt,
                                    int MBS, const int32_t *ctx, int B, int Hkv, int D, int BS, int64_t NB,
                                    cudaStream_t stream) {
    const int row_vecs = Hkv * D / 8;
    const dim3 grid{unsigned(MBS), unsigned(B), 1u};
    return launch_pdl(rebuild_meta_fp8_kernel, grid, dim3(64), 0, stream, reinterpret_cast<uint2 *>(kmin),
                      reinterpret_cast<uint2 *>(kmax), reinterpret_cast<const uint2 *>(kc), bt, MBS, ctx,
                      row_vecs, BS, NB);
}

}  // namespace pa
