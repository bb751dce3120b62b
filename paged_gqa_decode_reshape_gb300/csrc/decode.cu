// decode.cu -- GQA paged decode attention, dense and Quest-sparse (sm_103a).
//
// What it computes ("Ascend Kernel-to-Serving Pipeline", sections "GQA Paged
// Attention" and "Quest Sparse Attention"; split-KV per "18 e2e inference
// serving", section 4.1): for every sequence b and query head h,
//   out[b,h] = sum_t softmax_t(scale * q[b,h] . K_t) V_t
// over the sequence's tokens t < ctx_b (dense) or the tokens of its selected
// logical blocks (sparse), K/V gathered from the paged cache through the
// block table, query head h reading KV head h / G.
//
// How (GB300 design):
//  * Work list. Each (sequence, KV head) is a segment of items, one item per
//    KV block (dense: logical blocks 0..ceil(ctx/16)-1; sparse: the topk
//    selection entries). Segments are concatenated and the list is cut into
//    equal contiguous ranges, one per warp of a persistent grid (one or two
//    CTAs per SM). Every warp moves the same number of KV bytes whatever the
//    length mix; a warp's range touches at most a few segments.
//  * Data movement. Each warp owns an S-stage ring of shared-memory stages.
//    One lane issues two TMA tile loads per K and V block ([16 tokens x 64
//    dims] boxes of a 4-D tensor map over the whole pool, 128-byte swizzle)
//    with an L2 evict-first hint; the physical block number is a runtime TMA
//    coordinate. Stage completion is an mbarrier transaction count.
//  * Math. The GQA group's queries stay in registers as mma B fragments.
//    S^T = K Q^T and O^T += V^T P^T run on bf16 mma.sync (m16n8k16) with the
//    16 tokens of a block as the M dimension and the (up to 8) heads of the
//    group as N, so every K/V byte serves the whole group. Online softmax in
//    the log2 domain (running max, normaliser, rescaled accumulator), P
//    rounded to bf16 and transposed in registers with movmatrix.
//  * Masking. Tokens past ctx get score -inf and their V fragment lanes are
//    zeroed, so NaN/Inf garbage in unused slots never reaches the output.
//  * Combine. A warp that covers a whole segment writes bf16 output directly.
//    Otherwise each piece writes a normalised partial and its log2-sum-exp;
//    the last piece to arrive (atomic counter per segment) merges the pieces
//    with weights exp2(lse_s - max lse) and resets the counter to zero.
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

constexpr uint64_t kWaitLimitNs = 500ull * 1000ull * 1000ull;  // 0.5 s per mbarrier wait

template <int D>
struct DecodeCfg {
    static constexpr int BS = kBlockSize;
    static constexpr int KT = BS * D * 2;       // bytes of one K (or V) tile
    static constexpr int STAGE = 2 * KT;        // K + V
    static constexpr int NKK = D / 16;          // QK k-steps == PV m-tiles
    static constexpr int HALF = BS * 128;       // bytes of one 64-dim half tile
    static constexpr int PART = D * 8 + 8;      // floats per partial slot
    static constexpr int DPL = D / 32;          // dims per lane in the combine
    static constexpr int NW = 4;                // warps per CTA
    static constexpr int S = (D == 128) ? 6 : 8; // stages per warp
    static constexpr size_t smem_bytes(int B) {
        return 1024 + size_t(NW) * S * STAGE + size_t(NW) * S * 8 + size_t(B + 1) * 4;
    }
};

struct ItemInfo {
    int seg;   // b * Hkv + kvh, -1 past the range
    int phys;  // physical block, -1 if the block has no tokens to read
    int nv;    // valid tokens in the block (0..16)
};

template <int D, bool SPARSE>
__global__ void __launch_bounds__(DecodeCfg<D>::NW * 32, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D>;
    constexpr int BS = C::BS, NW = C::NW, S = C::S, NKK = C::NKK;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *base_ptr = smem_raw + (base - raw);
    const uint32_t bars = base + NW * S * C::STAGE;
    int32_t *pre = reinterpret_cast<int32_t *>(base_ptr + NW * S * C::STAGE + NW * S * 8);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, Hkv = a.Hkv, G = a.G;
    const int max_tok = a.MBS * BS;

    if (tid == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    // items per KV head of every sequence, then their prefix sum
    for (int b = tid; b < B; b += NW * 32) {
        const int c = min(max(__ldg(a.ctx + b), 0), max_tok);
        const int nblk = (c + BS - 1) / BS;
        pre[b + 1] = SPARSE ? (nblk > 0 ? a.topk : 0) : nblk;
    }
    if (tid == 0) pre[0] = 0;
    if (lane == 0) {
        for (int s = 0; s < S; ++s) mbar_init(bars + (warp * S + s) * 8, 1);
        fence_barrier_init();
    }
    __syncthreads();
    if (warp == 0) {
        int carry = 0;
        for (int b0 = 0; b0 < B; b0 += 32) {
            const int b = b0 + lane;
            int v = (b < B) ? pre[b + 1] : 0;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int u = __shfl_up_sync(0xffffffffu, v, o);
                if (lane >= o) v += u;
            }
            if (b < B) pre[b + 1] = carry + v;
            carry += __shfl_sync(0xffffffffu, v, 31);
        }
    }
    __syncthreads();

    // sequences with nothing to attend to get a zero output
    for (int idx = blockIdx.x * NW * 32 + tid; idx < B * a.Hq; idx += gridDim.x * NW * 32) {
        const int b = idx / a.Hq;
        if (pre[b + 1] == pre[b]) {
            uint4 *o = reinterpret_cast<uint4 *>(a.out + int64_t(idx) * D);
#pragma unroll
            for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
        }
    }

    const int64_t total = int64_t(Hkv) * pre[B];
    const int W = gridDim.x * NW;
    const int w = blockIdx.x * NW + warp;
    const int64_t L = (total + W - 1) / W;
    const int64_t pos0 = int64_t(w) * L;
    const int64_t pos1 = min(total, pos0 + L);
    if (pos0 >= pos1) return;  // no __syncthreads below this point
    const int n_items = int(pos1 - pos0);

    // where item k of this warp's range lives
    auto locate = [&](int k) -> ItemInfo {
        ItemInfo it{-1, -1, 0};
        if (k >= n_items) return it;
        const int64_t pos = pos0 + k;
        int lo = 0, hi = B;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (int64_t(Hkv) * pre[mid] <= pos) lo = mid; else hi = mid;
        }
        const int b = lo;
        const int n = pre[b + 1] - pre[b];
        const int64_t r = pos - int64_t(Hkv) * pre[b];
        const int kvh = int(r / n);
        const int i = int(r - int64_t(kvh) * n);
        const int c = min(max(__ldg(a.ctx + b), 0), max_tok);
        const int nblk = (c + BS - 1) / BS;
        const int j = SPARSE ? __ldg(a.sel + (int64_t(b) * Hkv + kvh) * a.topk + i) : i;
        it.seg = b * Hkv + kvh;
        if (j >= 0 && j < nblk) {
            const int ph = __ldg(a.bt + int64_t(b) * a.MBS + j);
            if (ph >= 0 && int64_t(ph) < a.NB) {
                it.phys = ph;
                it.nv = min(BS, c - j * BS);
            }
        }
        return it;
    };

    const uint32_t my_stages = base + warp * S * C::STAGE;
    const uint32_t my_bars = bars + warp * S * 8;
    const uint64_t policy = l2_policy_evict_first();

    // two 32-item windows of per-lane item info
    ItemInfo wa = locate(lane), wb = locate(32 + lane);
    int wbase = 0;
    auto item = [&](int k) -> ItemInfo {
        const bool first = k < wbase + 32;
        ItemInfo src = first ? wa : wb;
        ItemInfo r;
        r.seg = __shfl_sync(0xffffffffu, src.seg, k & 31);
        r.phys = __shfl_sync(0xffffffffu, src.phys, k & 31);
        r.nv = __shfl_sync(0xffffffffu, src.nv, k & 31);
        return r;
    };
    auto issue = [&](int k, const ItemInfo &it) {
        const int st = k % S;
        const uint32_t bar = my_bars + st * 8;
        if (it.phys >= 0) {
            const uint32_t dst = my_stages + st * C::STAGE;
            const int kvh = it.seg % Hkv;
            mbar_arrive_expect_tx(bar, C::STAGE);
#pragma unroll
            for (int hf = 0; hf < D / 64; ++hf) {
                tma_load_4d(dst + hf * C::HALF, &tm_k, bar, hf * 64, kvh, 0, it.phys, policy);
                tma_load_4d(dst + C::KT + hf * C::HALF, &tm_v, bar, hf * 64, kvh, 0, it.phys,
                            policy);
            }
        } else {
            mbar_arrive(bar);
        }
    };

    const int nprolog = min(S, n_items);
    for (int k = 0; k < nprolog; ++k) {
        const ItemInfo it = item(k);
        if (lane == 0) issue(k, it);
    }

    const int g = lane >> 2, q4 = lane & 3;
    uint32_t qb[NKK][2];
    float acc[NKK][4];
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    int cur_seg = -1;
    int64_t piece_begin = pos0;

    auto load_q = [&](int seg) {
        const int b = seg / Hkv, kvh = seg % Hkv;
        const bool hv = g < G;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            a.q + (int64_t(b) * a.Hq + kvh * G + (hv ? g : 0)) * D);
#pragma unroll
        for (int kk = 0; kk < NKK; ++kk) {
            qb[kk][0] = hv ? __ldg(qrow + 8 * kk + q4) : 0u;
            qb[kk][1] = hv ? __ldg(qrow + 8 * kk + 4 + q4) : 0u;
        }
#pragma unroll
        for (int mt = 0; mt < NKK; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    };

    // merge the pieces of segment `seg` (called by the last piece to arrive)
    auto combine = [&](int seg, int64_t s0, int64_t e0) {
        constexpr int DPL = C::DPL;
        const int b = seg / Hkv, kvh = seg % Hkv;
        const int w0 = int(s0 / L), w1 = int((e0 - 1) / L);
        float M[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) M[h] = -INFINITY;
        for (int ww = w0; ww <= w1; ++ww) {
            const float *ps = a.part + int64_t(seg + ww) * C::PART + D * 8;
#pragma unroll
            for (int h = 0; h < 8; ++h) M[h] = fmaxf(M[h], __ldcg(ps + h));
        }
        float o[DPL][8], ws[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            ws[h] = 0.f;
#pragma unroll
            for (int dd = 0; dd < DPL; ++dd) o[dd][h] = 0.f;
        }
        for (int ww = w0; ww <= w1; ++ww) {
            const float *ps = a.part + int64_t(seg + ww) * C::PART;
            float wt[8];
#pragma unroll
            for (int h = 0; h < 8; ++h) {
                const float lse = __ldcg(ps + D * 8 + h);
                wt[h] = (lse == -INFINITY) ? 0.f : fast_exp2(lse - M[h]);
                ws[h] += wt[h];
            }
#pragma unroll
            for (int dd = 0; dd < DPL; ++dd) {
                const float4 x0 = __ldcg(reinterpret_cast<const float4 *>(ps + (lane * DPL + dd) * 8));
                const float4 x1 = __ldcg(reinterpret_cast<const float4 *>(ps + (lane * DPL + dd) * 8 + 4));
                o[dd][0] += wt[0] * x0.x; o[dd][1] += wt[1] * x0.y;
                o[dd][2] += wt[2] * x0.z; o[dd][3] += wt[3] * x0.w;
                o[dd][4] += wt[4] * x1.x; o[dd][5] += wt[5] * x1.y;
                o[dd][6] += wt[6] * x1.z; o[dd][7] += wt[7] * x1.w;
            }
        }
#pragma unroll
        for (int h = 0; h < 8; ++h) {
            if (h >= G) break;
            const float inv = ws[h] > 0.f ? 1.f / ws[h] : 0.f;
            uint16_t *dst = a.out + (int64_t(b) * a.Hq + kvh * G + h) * D + lane * DPL;
            if (DPL == 4) {
                uint2 v;
                v.x = pack_bf16x2(o[0][h] * inv, o[1][h] * inv);
                v.y = pack_bf16x2(o[2 % DPL][h] * inv, o[3 % DPL][h] * inv);
                *reinterpret_cast<uint2 *>(dst) = v;
            } else {
                *reinterpret_cast<uint32_t *>(dst) = pack_bf16x2(o[0][h] * inv, o[1 % DPL][h] * inv);
            }
        }
    };

    auto finalize = [&](int seg, int64_t pb, int64_t pe) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
        const int b = seg / Hkv, kvh = seg % Hkv;
        const int n = pre[b + 1] - pre[b];
        const int64_t s0 = int64_t(Hkv) * pre[b] + int64_t(kvh) * n;
        const int64_t e0 = s0 + n;
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f;
        const float inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
        const int h0 = 2 * q4, h1 = 2 * q4 + 1;
        if (pb == s0 && pe == e0) {
            // the whole segment is in this piece: final bf16 output
            uint16_t *ob = a.out + (int64_t(b) * a.Hq + kvh * G) * D;
#pragma unroll
            for (int mt = 0; mt < NKK; ++mt) {
                const int d = 16 * mt + g;
                if (h0 < G) {
                    ob[h0 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][0] * inv0));
                    ob[h0 * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][2] * inv0));
                }
                if (h1 < G) {
                    ob[h1 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][1] * inv1));
                    ob[h1 * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][3] * inv1));
                }
            }
            return;
        }
        float *ps = a.part + int64_t(seg + w) * C::PART;
#pragma unroll
        for (int mt = 0; mt < NKK; ++mt) {
            const int d = 16 * mt + g;
            __stcg(reinterpret_cast<float2 *>(ps + d * 8 + h0),
                   make_float2(acc[mt][0] * inv0, acc[mt][1] * inv1));
            __stcg(reinterpret_cast<float2 *>(ps + (d + 8) * 8 + h0),
                   make_float2(acc[mt][2] * inv0, acc[mt][3] * inv1));
        }
        if (g == 0) {
            const float lse0 = l0 > 0.f ? m0 + log2f(l0) : -INFINITY;
            const float lse1 = l1 > 0.f ? m1 + log2f(l1) : -INFINITY;
            __stcg(reinterpret_cast<float2 *>(ps + D * 8 + h0), make_float2(lse0, lse1));
        }
        __threadfence();
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            const int npieces = int((e0 - 1) / L - s0 / L) + 1;
            const int old = atomicAdd(a.counters + seg, 1);
            last = (old == npieces - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        if (last) {
            __threadfence();
            combine(seg, s0, e0);
            if (lane == 0) a.counters[seg] = 0;
        }
    };

    const float scale_log2 = a.scale_log2;
    for (int i = 0; i < n_items; ++i) {
        if (i == wbase + 32) {
            wa = wb;
            wbase += 32;
            wb = locate(wbase + 32 + lane);
        }
        const ItemInfo it = item(i);
        if (it.seg != cur_seg) {
            if (cur_seg >= 0) finalize(cur_seg, piece_begin, pos0 + i);
            cur_seg = it.seg;
            piece_begin = pos0 + i;
            load_q(it.seg);
        }
        const int st = i % S;
        if (!mbar_wait_bounded(my_bars + st * 8, (i / S) & 1, kWaitLimitNs)) {
            // give up: record it, let the copies already issued land, leave
            if (lane == 0) atomicOr(a.status, kStatusTimeout);
            for (int k = i + 1; k < min(n_items, i + S); ++k)
                mbar_wait_bounded(my_bars + (k % S) * 8, (k / S) & 1, kWaitLimitNs);
            return;
        }
        const int nv = it.nv;
        if (nv > 0) {
            const uint32_t kb = my_stages + st * C::STAGE;
            const uint32_t vb = kb + C::KT;
            // ---- S^T = K Q^T (16 tokens x 8 heads)
            float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
            const int rk = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
            for (int kk = 0; kk < NKK; ++kk) {
                const int ch = ((kk & 3) << 1) + (lane >> 4);
                const uint32_t addr = kb + (kk >> 2) * C::HALF + rk * 128 + ((ch ^ (lane & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4(addr, a0, a1, a2, a3);
                if (kk & 1) mma_bf16(sb, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
                else mma_bf16(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
            }
            // ---- online softmax (log2 domain); rows g and g+8, heads h0 and h1
            const float x0 = (g < nv) ? (sa[0] + sb[0]) * scale_log2 : -INFINITY;
            const float x1 = (g < nv) ? (sa[1] + sb[1]) * scale_log2 : -INFINITY;
            const float x2 = (g + 8 < nv) ? (sa[2] + sb[2]) * scale_log2 : -INFINITY;
            const float x3 = (g + 8 < nv) ? (sa[3] + sb[3]) * scale_log2 : -INFINITY;
            float bm0 = fmaxf(x0, x2), bm1 = fmaxf(x1, x3);
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
                bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
                bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
            }
            const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
            const float r0 = (mn0 == -INFINITY) ? 0.f : mn0;
            const float r1 = (mn1 == -INFINITY) ? 0.f : mn1;
            const float al0 = fast_exp2(m0 - r0), al1 = fast_exp2(m1 - r1);
            const uint32_t p01 = pack_bf16x2(fast_exp2(x0 - r0), fast_exp2(x1 - r1));
            const uint32_t p23 = pack_bf16x2(fast_exp2(x2 - r0), fast_exp2(x3 - r1));
            l0 = l0 * al0 + (bf16_lo(p01) + bf16_lo(p23));
            l1 = l1 * al1 + (bf16_hi(p01) + bf16_hi(p23));
            m0 = mn0;
            m1 = mn1;
#pragma unroll
            for (int mt = 0; mt < NKK; ++mt) {
                acc[mt][0] *= al0;
                acc[mt][1] *= al1;
                acc[mt][2] *= al0;
                acc[mt][3] *= al1;
            }
            const uint32_t pb0 = movmatrix_trans(p01), pb1 = movmatrix_trans(p23);
            // ---- O^T += V^T P^T; V lanes of tokens >= nv zeroed
            uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
            if (nv < BS) {
                const int t0 = 2 * q4;
                mlo = (t0 < nv ? 0x0000ffffu : 0u) | (t0 + 1 < nv ? 0xffff0000u : 0u);
                mhi = (t0 + 8 < nv ? 0x0000ffffu : 0u) | (t0 + 9 < nv ? 0xffff0000u : 0u);
            }
            const int rv = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
            for (int mt = 0; mt < NKK; ++mt) {
                const int ch = ((mt & 3) << 1) + ((lane >> 3) & 1);
                const uint32_t addr = vb + (mt >> 2) * C::HALF + rv * 128 + ((ch ^ (lane & 7)) << 4);
                uint32_t a0, a1, a2, a3;
                ldsm_x4_trans(addr, a0, a1, a2, a3);
                mma_bf16(acc[mt], a0 & mlo, a1 & mlo, a2 & mhi, a3 & mhi, pb0, pb1);
            }
        }
        __syncwarp();
        const int k = i + S;
        if (k < n_items) {
            const ItemInfo nx = item(k);
            if (lane == 0) issue(k, nx);
        }
    }
    finalize(cur_seg, piece_begin, pos1);
}

template <int D, bool SPARSE>
cudaError_t launch_t(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                     cudaStream_t stream) {
    using C = DecodeCfg<D>;
    DecodeGeometry geo;
    cudaError_t e = decode_geometry(D, &geo);
    if (e != cudaSuccess) return e;
    const size_t smem = C::smem_bytes(a.B);
    decode_kernel<D, SPARSE><<<geo.grid, C::NW * 32, smem, stream>>>(tm_k, tm_v, a);
    return cudaGetLastError();
}

template <int D>
cudaError_t geometry_t(DecodeGeometry *g) {
    using C = DecodeCfg<D>;
    const size_t smem = C::smem_bytes(kMaxBatch);
    cudaError_t e;
    e = cudaFuncSetAttribute(decode_kernel<D, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(decode_kernel<D, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, int(smem));
    if (e != cudaSuccess) return e;
    int dev = 0, sms = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, false>, C::NW * 32, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    g->grid = sms * per_sm;
    g->warps = C::NW;
    g->workers = g->grid * C::NW;
    g->smem = smem;
    return cudaSuccess;
}

constexpr int kMaxDevices = 64;
DecodeGeometry g_geo[kMaxDevices][2];
bool g_geo_ok[kMaxDevices][2];

}  // namespace

cudaError_t decode_geometry(int head_dim, DecodeGeometry *g) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    const int idx = head_dim == 128 ? 1 : 0;
    if (!g_geo_ok[dev][idx]) {
        DecodeGeometry t{};
        e = head_dim == 128 ? geometry_t<128>(&t) : geometry_t<64>(&t);
        if (e != cudaSuccess) return e;
        g_geo[dev][idx] = t;
        g_geo_ok[dev][idx] = true;
    }
    *g = g_geo[dev][idx];
    return cudaSuccess;
}

size_t decode_workspace_bytes(int B, int Hkv, int head_dim, int workers) {
    const size_t segs = size_t(B) * Hkv;
    const size_t head = 256;                                        // status word + padding
    const size_t counters = (segs * 4 + 255) / 256 * 256;
    const size_t part = (segs + size_t(workers)) * size_t(head_dim * 8 + 8) * 4;
    return head + counters + part;
}

cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                          int head_dim, bool sparse, cudaStream_t stream) {
    if (head_dim == 128)
        return sparse ? launch_t<128, true>(tm_k, tm_v, a, stream)
                      : launch_t<128, false>(tm_k, tm_v, a, stream);
    return sparse ? launch_t<64, true>(tm_k, tm_v, a, stream)
                  : launch_t<64, false>(tm_k, tm_v, a, stream);
}

}  // namespace pa
