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

// ------------------------------------------------- per-block scales
//
// Each (physical block, KV head) has its own K and V scale, a power of two
// (0 while the block holds nothing). One call's write to a block, per head,
// for K and V alike: a = the largest finite |x| over the call's tokens in the
// block; e_call = the smallest e >= -126 with a <= 448 * 2^e; unless a token
// lands at offset 0 (the block restarts) and if the stored scale is 2^e_old,
// the new exponent is max(e_old, e_call), else e_call; when it grew, the
// block's codes at the offsets the call does not write are re-encoded with
// the factor 2^(e_old - e) (exact in the E4M3 normal range); the call's
// tokens are encoded with 2^e; the metadata follow the re-encoded codes.

// smallest e >= -126 with a <= 448 * 2^e (a >= 0): with a = m * 2^E,
// m in [0.5, 1), and 448 = 0.875 * 2^9, that is E - 9, plus 1 if m > 0.875
__device__ __forceinline__ int fit_exponent(float a) {
    if (!(a > 0.f)) return -126;
    int E = 0;
    const float m = frexpf(a, &E);
    return max(-126, E - 9 + (m > 0.875f ? 1 : 0));
}

__device__ __forceinline__ float pow2f(int e) {  // 2^e for -126 <= e <= 127
    return __uint_as_float(uint32_t(e + 127) << 23);
}

// 2^-d for d >= 0 (0 below the normal range: every code times it encodes to a zero)
__device__ __forceinline__ float shrink_factor(int d) { return d > 126 ? 0.f : pow2f(-d); }

// old and new exponent of one scale (e_old = e_new when there is no old scale)
__device__ __forceinline__ void block_exponents(bool reset, float stored, float amax, int &eo, int &en) {
    const int ec = fit_exponent(amax);
    int E = 0;
    const bool have = !reset && stored > 0.f;
    if (have) (void)frexpf(stored, &E);  // stored = 0.5 * 2^E
    en = have ? max(E - 1, ec) : ec;
    eo = have ? E - 1 : en;
}

// largest finite |x| of 8 bf16 elements (0 if none)
__device__ __forceinline__ float absmax8(const uint4 &x) {
    const uint32_t *w = reinterpret_cast<const uint32_t *>(&x);
    float m = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float a = fabsf(bf16_lo(w[i])), b = fabsf(bf16_hi(w[i]));
        if (a < INFINITY) m = fmaxf(m, a);
        if (b < INFINITY) m = fmaxf(m, b);
    }
    return m;
}

// 8 codes times f, re-encoded (nearest, ties to even; NaN as 0x7F)
__device__ __forceinline__ uint2 rescale8(const uint2 &c, float f) {
    const uint32_t w[2] = {c.x, c.y};
    uint32_t out[2];
#pragma unroll
    for (int i = 0; i < 2; ++i) {
        uint32_t word = 0;
#pragma unroll
        for (int j = 0; j < 2; ++j) {
            const uint32_t h = e4m3x2_to_f16x2(w[i] >> (16 * j));
            const float a = f16_lo(h) * f, b = f16_hi(h) * f;
            uint32_t pair = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
            if (a != a) pair = (pair & 0xff00u) | 0x7fu;
            if (b != b) pair = (pair & 0x00ffu) | 0x7f00u;
            word |= (pair & 0xffffu) << (16 * j);
        }
        out[i] = word;
    }
    return make_uint2(out[0], out[1]);
}

// One warp per token; the warp of the lowest-index token of the call in a
// physical block does all of the call's work on that block (the other
// warps return), so no two warps touch one block. Lane l handles the 8-dim
// vectors e = l, l + 32, ... of a token row (16 per KV head: head e / 16).
template <bool META>
__global__ void __launch_bounds__(32) write_fp8_block_kernel(
    uint2 *__restrict__ kc, uint8_t *__restrict__ vc, uint2 *__restrict__ kmin, uint2 *__restrict__ kmax,
    float *__restrict__ kbs, float *__restrict__ vbs, const uint4 *__restrict__ key,
    const uint4 *__restrict__ value, const int64_t *__restrict__ slots, int64_t T, int Hkv, int64_t NB) {
    constexpr int BS = kBlockSize, VPH = 16;  // head_dim 128: 16 vectors of 8 per head
    pdl_trigger();
    pdl_wait();
    const int64_t t = blockIdx.x;
    const int lane = threadIdx.x;
    if (t >= T) return;
    const int64_t s = __ldg(slots + t);
    if (s < 0 || s >= NB * BS) return;
    const int64_t p = s / BS;
    const int row_vecs = Hkv * VPH;
    // leadership, and the offsets of block p the call writes
    uint32_t wmask = 1u << (s % BS);
    int64_t first_later = -1;  // first 32-token chunk holding a later token in the block
    for (int64_t u0 = 0; u0 < T; u0 += 32) {
        const int64_t u = u0 + lane;
        const int64_t su = u < T ? __ldg(slots + u) : -1;
        const bool in_blk = su >= 0 && su < NB * BS && su / BS == p;
        if (__any_sync(0xffffffffu, in_blk && u < t)) return;  // not the leader
        const bool later = in_blk && u > t;
        wmask |= __reduce_or_sync(0xffffffffu, later ? (1u << (su % BS)) : 0u);
        if (first_later < 0 && __any_sync(0xffffffffu, later)) first_later = u0;
    }
    const bool reset = wmask & 1u;
    // the call's tokens in block p, in order (fn runs on the whole warp)
    auto for_members = [&](auto &&fn) {
        fn(t);
        if (first_later < 0) return;
        for (int64_t u0 = first_later; u0 < T; u0 += 32) {
            const int64_t u = u0 + lane;
            const int64_t su = u < T ? __ldg(slots + u) : -1;
            unsigned m = __ballot_sync(0xffffffffu, su >= 0 && su < NB * BS && su / BS == p && u > t);
            while (m) {
                const int bit = __ffs(m) - 1;
                m &= m - 1;
                fn(u0 + bit);
            }
        }
    };
    // byte positions of the written tokens in a row of the V layout
    uint32_t pmask = 0;
#pragma unroll
    for (int o = 0; o < BS; ++o)
        if (wmask & (1u << o)) pmask |= 1u << (4 * ((o & 7) >> 1) + 2 * (o >> 3) + (o & 1));

    for (int e0 = 0; e0 < row_vecs; e0 += 32) {
        const int e = e0 + lane;
        const bool act = e < row_vecs;
        const int h = min(e, row_vecs - 1) / VPH, d0 = (e % VPH) * 8;
        // the largest finite |k| and |v| of the call's tokens, per head
        float ak = 0.f, av = 0.f;
        for_members([&](int64_t u) {
            if (act) {
                ak = fmaxf(ak, absmax8(__ldg(key + u * row_vecs + e)));
                av = fmaxf(av, absmax8(__ldg(value + u * row_vecs + e)));
            }
        });
#pragma unroll
        for (int o = VPH / 2; o >= 1; o >>= 1) {  // the 16 lanes of one head
            ak = fmaxf(ak, __shfl_xor_sync(0xffffffffu, ak, o));
            av = fmaxf(av, __shfl_xor_sync(0xffffffffu, av, o));
        }
        const int64_t si = p * Hkv + h;
        const float sk_old = act ? kbs[si] : 0.f, sv_old = act ? vbs[si] : 0.f;
        __syncwarp();  // every lane has read the old scales before they are replaced
        int eko, ekn, evo, evn;
        block_exponents(reset, sk_old, ak, eko, ekn);
        block_exponents(reset, sv_old, av, evo, evn);
        if (act && e % VPH == 0) {
            kbs[si] = pow2f(ekn);
            vbs[si] = pow2f(evn);
        }
        // re-encode the block's other offsets when a scale grew
        if (act && ekn > eko) {
            const float f = shrink_factor(ekn - eko);
            for (int o = 0; o < BS; ++o)
                if (!(wmask & (1u << o))) {
                    uint2 *r = kc + (p * BS + o) * row_vecs + e;
                    *r = rescale8(*r, f);
                }
        }
        if (act && evn > evo) {
            const float f = shrink_factor(evn - evo);
            uint4 *rows = reinterpret_cast<uint4 *>(vc + ((p * Hkv + h) * 128 + d0) * 16);
            for (int dd = 0; dd < 8; ++dd) {
                const uint4 old = rows[dd];
                const uint2 lo = rescale8(make_uint2(old.x, old.y), f), hi = rescale8(make_uint2(old.z, old.w), f);
                const uint32_t nw[4] = {lo.x, lo.y, hi.x, hi.y}, ow[4] = {old.x, old.y, old.z, old.w};
                uint32_t res[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    uint32_t keep = 0;  // bytes of tokens the call writes stay as they are
#pragma unroll
                    for (int bb = 0; bb < 4; ++bb)
                        if (pmask & (1u << (4 * i + bb))) keep |= 0xffu << (8 * bb);
                    res[i] = (ow[i] & keep) | (nw[i] & ~keep);
                }
                rows[dd] = make_uint4(res[0], res[1], res[2], res[3]);
            }
        }
        // metadata: the stored min / max (re-encoded like the codes), or none on a restart
        uint2 lo = make_uint2(0u, 0u), hi = lo;
        bool have = false;
        if (META && act && !reset) {
            lo = kmin[p * row_vecs + e];
            hi = kmax[p * row_vecs + e];
            if (ekn > eko) {
                const float f = shrink_factor(ekn - eko);
                lo = rescale8(lo, f);
                hi = rescale8(hi, f);
            }
            have = true;
        }
        // the call's tokens, with the new scales
        const float ks = pow2f(ekn), vs = pow2f(evn);
        for_members([&](int64_t u) {
            if (!act) return;
            const int o = int(__ldg(slots + u) % BS);
            const int pos = 4 * ((o & 7) >> 1) + 2 * (o >> 3) + (o & 1);
            const uint2 kq = quantize8(__ldg(key + u * row_vecs + e), ks);
            kc[(p * BS + o) * row_vecs + e] = kq;
            const uint2 v = quantize8(__ldg(value + u * row_vecs + e), vs);
            uint8_t *vrow = vc + ((p * Hkv + h) * 128 + d0) * 16 + pos;
#pragma unroll
            for (int i = 0; i < 8; ++i) vrow[16 * i] = uint8_t(((i < 4 ? v.x : v.y) >> (8 * (i & 3))) & 0xffu);
            if (META) {
                if (!have) {
                    lo = kq;
                    hi = kq;
                    have = true;
                } else {
                    minmax8_e4m3(lo, hi, kq);
                }
            }
        });
        if (META && act) {
            kmin[p * row_vecs + e] = lo;
            kmax[p * row_vecs + e] = hi;
        }
        __syncwarp();
    }
}

}  // namespace

cudaError_t launch_write_fp8_block(uint8_t *kc, uint8_t *vc, uint8_t *kmin, uint8_t *kmax, float *k_bscale,
                                   float *v_bscale, const uint16_t *key, const uint16_t *value,
                                   const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                                   cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (D != 128 || BS != kBlockSize) return cudaErrorInvalidValue;
    auto *kfn = kmin ? write_fp8_block_kernel<true> : write_fp8_block_kernel<false>;
    return launch_pdl(kfn, dim3(unsigned(T)), dim3(32), 0, stream, reinterpret_cast<uint2 *>(kc), vc,
                      reinterpret_cast<uint2 *>(kmin), reinterpret_cast<uint2 *>(kmax), k_bscale, v_bscale,
                      reinterpret_cast<const uint4 *>(key), reinterpret_cast<const uint4 *>(value), slots, T,
                      Hkv, NB);
}

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
