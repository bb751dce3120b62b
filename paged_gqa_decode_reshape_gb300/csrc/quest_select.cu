// quest_select.cu -- Quest block scoring and top-K selection (sm_103a).
//
// "Ascend Kernel-to-Serving Pipeline", section "Quest Sparse Attention": score
// the logical blocks cheaply, keep the top-K, attend over those only. The
// score of logical block j of sequence b for KV head g is the upper bound
//     sum_{h in group g} sum_d max(q[b,h,d] * kmin[p,g,d], q[b,h,d] * kmax[p,g,d])
// with p = block_tables[b][j]; ties in the top-K go to the lower block index.
//
// Score evaluation (fp32, one fixed order shared with the CPU oracle, since
// the scores decide an integer set): max(q*mn, q*mx) = q+ * mx + q- * mn with
// q+ = max(q, 0), q- = min(q, 0), so with P_d = sum_h q+ and N_d = sum_h q-
// (h ascending from +0) every block costs two products and one add per
// dimension: t_d = fl(fl(P_d * mx_d) + fl(N_d * mn_d)). Lane l of a warp sums
// t_d over its D/32 consecutive dims left to right; the 32 lane sums are
// combined by a xor butterfly (16, 8, 4, 2, 1). No FMA contraction (the
// products and sums are explicit __fmul_rn / __fadd_rn).
//
// Work split: a persistent grid; the (sequence, KV head, 8-block chunk) list
// is cut into equal contiguous ranges, one per warp; a warp reads each
// block's two metadata rows with one 8-byte (D=128) load per lane, i.e. 256
// contiguous bytes per row per warp, a whole chunk in flight.
//
// Top-K: one CTA per (sequence, KV head): a radix select over the
// totalOrder keys of the scores (digits of up to 8 bits, from the highest bit
// where the row's keys differ) finds the K-th largest key; blocks above it,
// then the lowest-index blocks equal to it, are written in ascending block
// order (cta_topk_threshold, cta_topk_emit).
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

constexpr int kTopkThreads = 256;

// Persistent grid: the list of (sequence, KV head, chunk of kChunk logical
// blocks) is cut into equal contiguous ranges, one per warp. A warp walks its
// range: per chunk one round trip for the block-table entries (one per lane)
// and one for both metadata rows of all the chunk's blocks; the query group's
// P/N sums are formed once per (sequence, KV head).
constexpr int kChunk = 8;
constexpr int kScoreThreads = 256;

// F8: the metadata are E4M3 codes (one byte per element, decoded exactly);
// the score is the same fp32 expression of the decoded values. With
// per-block scales (kbs [NB][Hkv], else null) the block's score is then
// multiplied by its K scale (one fp32 product, exact for a power of two).
//
// With the step's write (bf16, wr.key not null): the warp whose chunk holds
// block (ctx_b - 1) / BS of sequence b writes token b's KV-head slice into
// the cache when wr.slots[b] is the slot of position ctx_b - 1, and updates
// that block's metadata (reset at offset 0, else merged), before it loads
// the chunk's metadata; the loads then see the update (same lane, same
// address, no read-only cache path).
template <int D, bool F8>
__global__ void __launch_bounds__(kScoreThreads, 4) quest_score_kernel(
    float *__restrict__ scores, const uint16_t *__restrict__ q, const void *kmin_v,
    const void *kmax_v, const float *__restrict__ kbs, const int32_t *__restrict__ bt,
    int MBS, const int32_t *__restrict__ ctx, int B, int Hq, int Hkv, int BS, int64_t NB, ScoreWrite wr) {
    static_assert(!F8 || D == 128, "E4M3 metadata: head_dim 128");
    const uint16_t *kmin = static_cast<const uint16_t *>(kmin_v);
    const uint16_t *kmax = static_cast<const uint16_t *>(kmax_v);
    constexpr int C = D / 32;  // dims per lane
    constexpr int CW = C / 2;  // 32-bit words per lane per row
    extern __shared__ int32_t pre[];  // [B+1] chunk prefix per KV head
    pdl_trigger();
    // The context lengths and the first chunk's block-table entries are the
    // caller's inputs, which no kernel of this library writes: they are read
    // while the previous kernel in the stream finishes. Everything else (q,
    // the metadata, the scores, the step's write) waits for it.
    const int tid = threadIdx.x, lane = tid & 31;
    const int G = Hq / Hkv;
    const int max_tok = MBS * BS;
    {
        // L2 prefetch hints (no registers held): the block table and the
        // queries, a 128-byte line per thread of the grid. L2 is coherent
        // with the previous kernel's writes, so hints may precede the wait.
        const int64_t nthr = int64_t(gridDim.x) * kScoreThreads;
        const int64_t gt = int64_t(blockIdx.x) * kScoreThreads + tid;
        for (int64_t off = gt * 32; off < int64_t(B) * MBS; off += nthr * 32) prefetch_l2(bt + off);
        for (int64_t off = gt * 64; off < int64_t(B) * Hq * D; off += nthr * 64) prefetch_l2(q + off);
    }
    for (int b = tid; b < B; b += kScoreThreads) {
        const int c = min(max(__ldg(ctx + b), 0), max_tok);
        pre[b + 1] = ((c + BS - 1) / BS + kChunk - 1) / kChunk;
    }
    if (tid == 0) pre[0] = 0;
    __syncthreads();
    if (tid < 32) {
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
    const int64_t total = int64_t(Hkv) * pre[B];
    const int64_t W = int64_t(gridDim.x) * (kScoreThreads / 32);
    const int64_t w = int64_t(blockIdx.x) * (kScoreThreads / 32) + (tid >> 5);
    const int64_t R = (total + W - 1) / W;
    int64_t id = w * R;
    const int64_t id1 = min(total, id + R);
    if (id >= id1) {
        pdl_wait();
        return;
    }
    // locate the first chunk
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (int64_t(Hkv) * pre[mid] <= id) lo = mid; else hi = mid;
    }
    int b = lo;
    int nch = pre[b + 1] - pre[b];
    int kvh = int((id - int64_t(Hkv) * pre[b]) / nch);
    int ch = int(id - int64_t(Hkv) * pre[b] - int64_t(kvh) * nch);
    // block-table entries of chunk (b, ch), one per lane
    auto chunk_phys = [&](int bb, int cc) -> int {
        const int nb = (min(max(__ldg(ctx + bb), 0), max_tok) + BS - 1) / BS;
        const int j = cc * kChunk + lane;
        return (lane < kChunk && j < nb) ? __ldg(bt + int64_t(bb) * MBS + j) : -1;
    };
    int ph_first = chunk_phys(b, ch);
    if (ph_first >= 0 && int64_t(ph_first) < NB) {
        // the first chunk's metadata rows into L2 while the previous kernel
        // finishes (lane u: block u's two rows)
        constexpr int EB = F8 ? 1 : 2;  // bytes per element
        const int64_t off = (int64_t(ph_first) * Hkv + kvh) * D * EB;
#pragma unroll
        for (int x = 0; x < D * EB; x += 128) {
            prefetch_l2(static_cast<const uint8_t *>(kmin_v) + off + x);
            prefetch_l2(static_cast<const uint8_t *>(kmax_v) + off + x);
        }
    }
    bool first = true;
    pdl_wait();
    int pn_seg = -1;
    float P[C], N[C];
    for (; id < id1; ++id) {
        const int c = min(max(__ldg(ctx + b), 0), max_tok);
        const int nblk = (c + BS - 1) / BS;
        const int j0 = ch * kChunk;
        const int cnt = min(kChunk, nblk - j0);
        const int ph_l = first ? ph_first : chunk_phys(b, ch);
        first = false;
        if (b * Hkv + kvh != pn_seg) {
            // P_d = sum_h max(q, 0), N_d = sum_h min(q, 0), h ascending from +0
            pn_seg = b * Hkv + kvh;
#pragma unroll
            for (int cc = 0; cc < C; ++cc) {
                P[cc] = 0.f;
                N[cc] = 0.f;
            }
            // the group's query rows, QB loads in flight before their sums
            constexpr int QB = 4;
            for (int g0 = 0; g0 < G; g0 += QB) {
                uint32_t qw[QB][CW];
#pragma unroll
                for (int i = 0; i < QB; ++i) {
                    if (g0 + i >= G) break;
                    const uint16_t *qr = q + (int64_t(b) * Hq + int64_t(kvh) * G + g0 + i) * D + lane * C;
                    if (C == 4) {
                        const uint2 v2 = __ldg(reinterpret_cast<const uint2 *>(qr));
                        qw[i][0] = v2.x;
                        qw[i][CW - 1] = v2.y;
                    } else {
                        qw[i][0] = __ldg(reinterpret_cast<const uint32_t *>(qr));
                    }
                }
#pragma unroll
                for (int i = 0; i < QB; ++i) {
                    if (g0 + i >= G) break;
#pragma unroll
                    for (int cc = 0; cc < C; ++cc) {
                        const float v = (cc & 1) ? bf16_hi(qw[i][cc >> 1]) : bf16_lo(qw[i][cc >> 1]);
                        P[cc] = __fadd_rn(P[cc], v > 0.f ? v : 0.f);
                        N[cc] = __fadd_rn(N[cc], v < 0.f ? v : 0.f);
                    }
                }
            }
        }
        if constexpr (!F8) {
            const int jl = nblk - 1;  // the block holding the new token
            if (wr.key && jl >= j0 && jl < j0 + cnt) {
                const int ph = __shfl_sync(0xffffffffu, ph_l, jl - j0);
                const int o = (c - 1) % BS;
                if (ph >= 0 && int64_t(ph) < NB && __ldg(wr.slots + b) == int64_t(ph) * BS + o) {
                    const int64_t src = (int64_t(b) * Hkv + kvh) * D + lane * C;
                    const int64_t dst = ((int64_t(ph) * BS + o) * Hkv + kvh) * D + lane * C;
                    const int64_t m = (int64_t(ph) * Hkv + kvh) * D + lane * C;
                    uint32_t kx[CW], vx[CW], lo[CW], hi[CW];
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
                        kx[i] = __ldg(reinterpret_cast<const uint32_t *>(wr.key + src) + i);
                        vx[i] = __ldg(reinterpret_cast<const uint32_t *>(wr.value + src) + i);
                        lo[i] = kx[i];
                        hi[i] = kx[i];
                        if (o != 0) {
                            lo[i] = __ldcg(reinterpret_cast<const uint32_t *>(wr.kmin + m) + i);
                            hi[i] = __ldcg(reinterpret_cast<const uint32_t *>(wr.kmax + m) + i);
                            minmax_bf16x2(lo[i], hi[i], kx[i]);
                        }
                    }
#pragma unroll
                    for (int i = 0; i < CW; ++i) {
                        reinterpret_cast<uint32_t *>(wr.kc + dst)[i] = kx[i];
                        reinterpret_cast<uint32_t *>(wr.vc + dst)[i] = vx[i];
                        reinterpret_cast<uint32_t *>(wr.kmin + m)[i] = lo[i];
                        reinterpret_cast<uint32_t *>(wr.kmax + m)[i] = hi[i];
                    }
                }
            }
        }
        uint32_t mnv[kChunk][CW], mxv[kChunk][CW];
        bool ok[kChunk];
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            const int ph = __shfl_sync(0xffffffffu, ph_l, u);
            ok[u] = (u < cnt) && ph >= 0 && int64_t(ph) < NB;
            const int64_t off = (int64_t(ok[u] ? ph : 0) * Hkv + kvh) * D + lane * C;
            if constexpr (F8) {  // C = 4 codes per lane per row
                mnv[u][0] = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(kmin_v) + off));
                mxv[u][0] = __ldg(reinterpret_cast<const uint32_t *>(static_cast<const uint8_t *>(kmax_v) + off));
            } else if (C == 4) {
                const uint2 a2 = __ldcg(reinterpret_cast<const uint2 *>(kmin + off));
                const uint2 b2 = __ldcg(reinterpret_cast<const uint2 *>(kmax + off));
                mnv[u][0] = a2.x;
                mnv[u][CW - 1] = a2.y;
                mxv[u][0] = b2.x;
                mxv[u][CW - 1] = b2.y;
            } else {
                mnv[u][0] = __ldcg(reinterpret_cast<const uint32_t *>(kmin + off));
                mxv[u][0] = __ldcg(reinterpret_cast<const uint32_t *>(kmax + off));
            }
        }
        // per-block K scale of block j0 + lane (E4M3 cache with block scales)
        const float bsc = (F8 && kbs && lane < cnt && ph_l >= 0 && int64_t(ph_l) < NB)
                              ? __ldg(kbs + int64_t(ph_l) * Hkv + kvh)
                              : 1.f;
        float mine = -INFINITY;  // lane u keeps block j0 + u's score
#pragma unroll
        for (int u = 0; u < kChunk; ++u) {
            float acc = 0.f;
#pragma unroll
            for (int cc = 0; cc < C; ++cc) {
                float mn, mx;
                if constexpr (F8) {
                    const uint32_t hmn = e4m3x2_to_f16x2(mnv[u][0] >> (16 * (cc >> 1)));
                    const uint32_t hmx = e4m3x2_to_f16x2(mxv[u][0] >> (16 * (cc >> 1)));
                    mn = (cc & 1) ? f16_hi(hmn) : f16_lo(hmn);
                    mx = (cc & 1) ? f16_hi(hmx) : f16_lo(hmx);
                } else {
                    const uint32_t wmn = mnv[u][cc >> 1], wmx = mxv[u][cc >> 1];
                    mn = (cc & 1) ? bf16_hi(wmn) : bf16_lo(wmn);
                    mx = (cc & 1) ? bf16_hi(wmx) : bf16_lo(wmx);
                }
                const float t = __fadd_rn(__fmul_rn(P[cc], mx), __fmul_rn(N[cc], mn));
                acc = (cc == 0) ? t : __fadd_rn(acc, t);
            }
#pragma unroll
            for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
            if (lane == u) mine = ok[u] ? acc : -INFINITY;
        }
        if (F8 && kbs && lane < cnt && mine != -INFINITY) mine = __fmul_rn(mine, bsc);
        if (lane < cnt) scores[(int64_t(b) * Hkv + kvh) * MBS + j0 + lane] = mine;
        // next chunk
        if (++ch == nch) {
            ch = 0;
            if (++kvh == Hkv) {
                kvh = 0;
                do {
                    ++b;
                } while (b < B && pre[b + 1] == pre[b]);
                if (b >= B) break;
                nch = pre[b + 1] - pre[b];
            }
        }
    }
}

// Keys cached in shared memory (12 KiB; longer rows are re-read from L2 on
// every pass): small, so that a top-K CTA fits on an SM beside a decode CTA.
constexpr int kTopkSmemKeys = 3072;

__global__ void __launch_bounds__(kTopkThreads, 4) quest_topk_kernel(
    int32_t *__restrict__ sel, const float *__restrict__ scores, int MBS,
    const int32_t *__restrict__ ctx, int Hkv, int BS, int topk) {
    __shared__ int hist[256];
    __shared__ int red[2 * kTopkThreads / 32 + 3];
    __shared__ uint32_t keys[kTopkSmemKeys];
    pdl_trigger();
    const int seg = blockIdx.x;
    const int b = seg / Hkv;
    const int tid = threadIdx.x;
    // the context length is the caller's input: read while the score kernel finishes
    const int c = min(max(__ldg(ctx + b), 0), MBS * BS);
    const int n = (c + BS - 1) / BS;
    pdl_wait();
    const float *srow = scores + int64_t(seg) * MBS;
    int32_t *out = sel + int64_t(seg) * topk;
    if (n <= topk) {
        for (int i = tid; i < topk; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    // totalOrder keys of the segment's scores: in shared memory when they fit
    const bool cached = n <= kTopkSmemKeys;
    if (cached) cta_load_keys<kTopkThreads>(keys, srow, n);
    __syncthreads();
    auto key_of = [&](int j) -> uint32_t { return cached ? keys[j] : f32_order_key(__ldcg(srow + j)); };
    uint32_t thr;
    int keq;
    cta_topk_threshold<kTopkThreads>(key_of, n, topk, hist, red, thr, keq);
    cta_topk_emit<kTopkThreads>(key_of, n, thr, keq, red, [&](int r, int j) { out[r] = j; });
}

template <int D, bool F8>
cudaError_t launch_score(float *scores, const uint16_t *q, const void *kmin, const void *kmax,
                         const float *kbs, const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hq,
                         int Hkv, int BS, int64_t NB, cudaStream_t stream, const ScoreWrite *write) {
    // persistent grid, every SM full (computed once, thread-safe; the same on
    // every GPU of a node)
    static const int grid = [] {
        int dev = 0, sms = 0, per_sm = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quest_score_kernel<D, F8>, kScoreThreads,
                                                          size_t(kMaxBatch + 1) * 4) != cudaSuccess)
            return 0;
        return sms * (per_sm < 1 ? 1 : per_sm);
    }();
    if (grid == 0) return cudaErrorInvalidConfiguration;
    const size_t smem = size_t(B + 1) * 4;
    ScoreWrite wr{};
    if (write) wr = *write;
    return launch_pdl(quest_score_kernel<D, F8>, dim3(grid), dim3(kScoreThreads), smem, stream, scores, q,
                      kmin, kmax, kbs, bt, MBS, ctx, B, Hq, Hkv, BS, NB, wr);
}

}  // namespace

cudaError_t launch_quest_scores(float *scores, const uint16_t *q, const void *kmin, const void *kmax,
                                const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hq, int Hkv, int D,
                                int BS, int64_t NB, cudaStream_t stream, bool fp8, const float *k_bscale,
                                const ScoreWrite *write) {
    if (fp8) {
        if (D != 128 || write) return cudaErrorInvalidValue;
        return launch_score<128, true>(scores, q, kmin, kmax, k_bscale, bt, MBS, ctx, B, Hq, Hkv, BS, NB,
                                       stream, nullptr);
    }
    return D == 128 ? launch_score<128, false>(scores, q, kmin, kmax, nullptr, bt, MBS, ctx, B, Hq, Hkv, BS, NB,
                                               stream, write)
                    : launch_score<64, false>(scores, q, kmin, kmax, nullptr, bt, MBS, ctx, B, Hq, Hkv, BS, NB,
                                              stream, write);
}

cudaError_t launch_quest_select(int32_t *sel, float *scores, const uint16_t *q, const void *kmin,
                                const void *kmax, const int32_t *bt, int MBS, const int32_t *ctx,
                                int B, int Hq, int Hkv, int D, int BS, int64_t NB, int topk,
                                cudaStream_t stream, bool fp8, const float *k_bscale, const ScoreWrite *write) {
    const cudaError_t e = launch_quest_scores(scores, q, kmin, kmax, bt, MBS, ctx, B, Hq, Hkv, D, BS, NB, stream,
                                              fp8, k_bscale, write);
    if (e != cudaSuccess) return e;
    return launch_pdl(quest_topk_kernel, dim3(unsigned(B) * unsigned(Hkv)), dim3(kTopkThreads), 0, stream,
                      sel, static_cast<const float *>(scores), MBS, ctx, Hkv, BS, topk);
}

}  // namespace pa
