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
// Work split: the (sequence, KV head, block) list is cut into equal contiguous
// ranges, one per warp of a persistent grid; a warp reads each block's two
// metadata rows with one 8-byte (D=128) load per lane, i.e. 256 contiguous
// bytes per row per warp, four blocks in flight per step.
//
// Top-K: one CTA per (sequence, KV head): a 4-pass, 8-bit radix select over
// the totalOrder keys of the scores finds the K-th largest key; blocks above
// it, then the lowest-index blocks equal to it, are written in ascending
// block order.
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

constexpr int kScoreWarps = 8;
constexpr int kTopkThreads = 256;

template <int D>
__global__ void __launch_bounds__(kScoreWarps * 32) quest_score_kernel(
    float *__restrict__ scores, const uint16_t *__restrict__ q, const uint16_t *__restrict__ kmin,
    const uint16_t *__restrict__ kmax, const int32_t *__restrict__ bt, int MBS,
    const int32_t *__restrict__ ctx, int B, int Hq, int Hkv, int BS, int64_t NB) {
    constexpr int C = D / 32;  // dims per lane
    extern __shared__ int32_t pre[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int G = Hq / Hkv;
    const int max_tok = MBS * BS;
    for (int b = tid; b < B; b += blockDim.x) {
        const int c = min(max(__ldg(ctx + b), 0), max_tok);
        pre[b + 1] = (c + BS - 1) / BS;
    }
    if (tid == 0) pre[0] = 0;
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

    const int64_t total = int64_t(Hkv) * pre[B];
    const int W = gridDim.x * kScoreWarps;
    const int w = blockIdx.x * kScoreWarps + warp;
    const int64_t L = (total + W - 1) / W;
    int64_t pos = int64_t(w) * L;
    const int64_t pos1 = min(total, pos + L);
    if (pos >= pos1) return;

    // locate the first item
    int lo = 0, hi = B;
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (int64_t(Hkv) * pre[mid] <= pos) lo = mid; else hi = mid;
    }
    int b = lo;
    int n = pre[b + 1] - pre[b];
    int64_t r = pos - int64_t(Hkv) * pre[b];
    int kvh = int(r / n);
    int j = int(r - int64_t(kvh) * n);

    while (pos < pos1) {
        const int j_end = int(min(int64_t(n), int64_t(j) + (pos1 - pos)));
        const int32_t *bt_row = bt + int64_t(b) * MBS;
        float *srow = scores + (int64_t(b) * Hkv + kvh) * MBS;
        // first chunk's block-table entries, in flight while P/N are formed
        int ph_next = (j + lane < j_end) ? __ldg(bt_row + j + lane) : -1;
        // P_d, N_d of this (b, kvh) for this lane's dims
        float P[C], N[C];
#pragma unroll
        for (int c = 0; c < C; ++c) {
            P[c] = 0.f;
            N[c] = 0.f;
        }
        for (int gg = 0; gg < G; ++gg) {
            const uint16_t *qr = q + (int64_t(b) * Hq + int64_t(kvh) * G + gg) * D + lane * C;
            uint32_t qw[C / 2];
            if (C == 4) {
                const uint2 v2 = __ldg(reinterpret_cast<const uint2 *>(qr));
                qw[0] = v2.x;
                qw[C / 2 - 1] = v2.y;
            } else {
                qw[0] = __ldg(reinterpret_cast<const uint32_t *>(qr));
            }
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float v = (c & 1) ? bf16_hi(qw[c >> 1]) : bf16_lo(qw[c >> 1]);
                P[c] = __fadd_rn(P[c], v > 0.f ? v : 0.f);
                N[c] = __fadd_rn(N[c], v < 0.f ? v : 0.f);
            }
        }
        for (int j0 = j; j0 < j_end; j0 += 32) {
            // physical blocks of up to 32 items, one per lane
            const int ph_l = ph_next;
            if (j0 + 32 < j_end) ph_next = (j0 + 32 + lane < j_end) ? __ldg(bt_row + j0 + 32 + lane) : -1;
            const int cnt = min(32, j_end - j0);
            for (int i0 = 0; i0 < cnt; i0 += 4) {
                float sc[4];
                uint32_t mnv[4][C / 2 > 0 ? C / 2 : 1], mxv[4][C / 2 > 0 ? C / 2 : 1];
                bool ok[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const int ph = __shfl_sync(0xffffffffu, ph_l, (i0 + u) & 31);
                    ok[u] = (i0 + u < cnt) && ph >= 0 && int64_t(ph) < NB;
                    const int64_t off = (int64_t(ok[u] ? ph : 0) * Hkv + kvh) * D + lane * C;
                    if (C == 4) {
                        const uint2 a2 = __ldg(reinterpret_cast<const uint2 *>(kmin + off));
                        const uint2 b2 = __ldg(reinterpret_cast<const uint2 *>(kmax + off));
                        mnv[u][0] = a2.x; mnv[u][C / 2 - 1] = a2.y;
                        mxv[u][0] = b2.x; mxv[u][C / 2 - 1] = b2.y;
                    } else {
                        mnv[u][0] = __ldg(reinterpret_cast<const uint32_t *>(kmin + off));
                        mxv[u][0] = __ldg(reinterpret_cast<const uint32_t *>(kmax + off));
                    }
                }
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    float acc = 0.f;
#pragma unroll
                    for (int c = 0; c < C; ++c) {
                        const uint32_t wmn = mnv[u][c >> 1], wmx = mxv[u][c >> 1];
                        const float mn = (c & 1) ? bf16_hi(wmn) : bf16_lo(wmn);
                        const float mx = (c & 1) ? bf16_hi(wmx) : bf16_lo(wmx);
                        const float t = __fadd_rn(__fmul_rn(P[c], mx), __fmul_rn(N[c], mn));
                        acc = (c == 0) ? t : __fadd_rn(acc, t);
                    }
#pragma unroll
                    for (int o = 16; o >= 1; o >>= 1) acc = __fadd_rn(acc, __shfl_xor_sync(0xffffffffu, acc, o));
                    sc[u] = ok[u] ? acc : -INFINITY;
                }
                if (lane < 4 && i0 + lane < cnt) {
                    float v = sc[0];
#pragma unroll
                    for (int u = 1; u < 4; ++u)
                        if (lane == u) v = sc[u];
                    srow[j0 + i0 + lane] = v;
                }
            }
        }
        pos += j_end - j;
        // next segment
        j = 0;
        if (++kvh == Hkv) {
            kvh = 0;
            do {
                ++b;
            } while (b < B && pre[b + 1] == pre[b]);
            if (b >= B) break;
            n = pre[b + 1] - pre[b];
        }
    }
}

// block-wide exclusive scan of a 0/1 flag (kTopkThreads threads)
__device__ __forceinline__ int block_rank(bool flag, int *warp_cnt, int &total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const unsigned bal = __ballot_sync(0xffffffffu, flag);
    const int in_warp = __popc(bal & ((1u << lane) - 1u));
    __syncthreads();
    if (lane == 0) warp_cnt[warp] = __popc(bal);
    __syncthreads();
    int before = 0;
    total = 0;
#pragma unroll
    for (int w = 0; w < kTopkThreads / 32; ++w) {
        const int c = warp_cnt[w];
        before += (w < warp) ? c : 0;
        total += c;
    }
    return before + in_warp;
}

constexpr int kTopkSmemKeys = 8192;  // keys cached in shared memory (32 KiB)

__global__ void __launch_bounds__(kTopkThreads) quest_topk_kernel(
    int32_t *__restrict__ sel, const float *__restrict__ scores, int MBS,
    const int32_t *__restrict__ ctx, int Hkv, int BS, int topk) {
    __shared__ int hist[256];
    __shared__ int warp_cnt[kTopkThreads / 32];
    __shared__ int sh_digit, sh_above;
    __shared__ uint32_t keys[kTopkSmemKeys];
    const int seg = blockIdx.x;
    const int b = seg / Hkv;
    const int tid = threadIdx.x, lane = tid & 31;
    const int c = min(max(__ldg(ctx + b), 0), MBS * BS);
    const int n = (c + BS - 1) / BS;
    const float *srow = scores + int64_t(seg) * MBS;
    int32_t *out = sel + int64_t(seg) * topk;
    if (n <= topk) {
        for (int i = tid; i < topk; i += kTopkThreads) out[i] = i < n ? i : -1;
        return;
    }
    // totalOrder keys of the segment's scores: in shared memory when they fit
    const bool cached = n <= kTopkSmemKeys;
    if (cached)
        for (int j = tid; j < n; j += kTopkThreads) keys[j] = f32_order_key(__ldcg(srow + j));
    auto key_of = [&](int j) -> uint32_t { return cached ? keys[j] : f32_order_key(__ldcg(srow + j)); };
    uint32_t prefix = 0, mask = 0;
    int k = topk;
    for (int shift = 24; shift >= 0; shift -= 8) {
        hist[tid] = 0;  // kTopkThreads == 256 bins
        __syncthreads();
        for (int j = tid; j < n; j += kTopkThreads) {
            const uint32_t u = key_of(j);
            if ((u & mask) == prefix) atomicAdd(&hist[(u >> shift) & 255u], 1);
        }
        __syncthreads();
        if (tid < 32) {
            // lane l holds digits 255-8l .. 248-8l (descending)
            int cnt[8], s = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                cnt[i] = hist[255 - 8 * lane - i];
                s += cnt[i];
            }
            int incl = s;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            int before = incl - s;
            if (before < k && k <= incl) {
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    if (before + cnt[i] >= k) {
                        sh_digit = 255 - 8 * lane - i;
                        sh_above = before;
                        break;
                    }
                    before += cnt[i];
                }
            }
        }
        __syncthreads();
        prefix |= uint32_t(sh_digit) << shift;
        mask |= 0xffu << shift;
        k -= sh_above;
        __syncthreads();
    }
    // prefix is the K-th largest key; take every key above it and the k
    // lowest-index keys equal to it, in ascending block order
    int carry_eq = 0, carry_pos = 0;
    for (int j0 = 0; j0 < n; j0 += kTopkThreads) {
        const int j = j0 + tid;
        const uint32_t u = j < n ? key_of(j) : 0u;
        const bool gt = j < n && u > prefix;
        const bool eq = j < n && u == prefix;
        int tot_eq;
        const int r_eq = block_rank(eq, warp_cnt, tot_eq) + carry_eq;
        const bool take = gt || (eq && r_eq < k);
        int tot_take;
        const int r_take = block_rank(take, warp_cnt, tot_take) + carry_pos;
        if (take) out[r_take] = j;
        carry_eq += tot_eq;
        carry_pos += tot_take;
    }
}

template <int D>
cudaError_t launch_score(float *scores, const uint16_t *q, const uint16_t *kmin,
                         const uint16_t *kmax, const int32_t *bt, int MBS, const int32_t *ctx,
                         int B, int Hq, int Hkv, int BS, int64_t NB, cudaStream_t stream) {
    const size_t smem = size_t(B + 1) * 4;
    int dev = 0, sms = 0, per_sm = 0;
    cudaError_t e;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quest_score_kernel<D>,
                                                      kScoreWarps * 32, smem);
    if (e != cudaSuccess) return e;
    per_sm = per_sm < 1 ? 1 : per_sm;
    quest_score_kernel<D><<<sms * per_sm, kScoreWarps * 32, smem, stream>>>(
        scores, q, kmin, kmax, bt, MBS, ctx, B, Hq, Hkv, BS, NB);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quest_select(int32_t *sel, float *scores, const uint16_t *q,
                                const uint16_t *kmin, const uint16_t *kmax, const int32_t *bt,
                                int MBS, const int32_t *ctx, int B, int Hq, int Hkv, int D, int BS,
                                int64_t NB, int topk, cudaStream_t stream) {
    cudaError_t e = D == 128
        ? launch_score<128>(scores, q, kmin, kmax, bt, MBS, ctx, B, Hq, Hkv, BS, NB, stream)
        : launch_score<64>(scores, q, kmin, kmax, bt, MBS, ctx, B, Hq, Hkv, BS, NB, stream);
    if (e != cudaSuccess) return e;
    quest_topk_kernel<<<unsigned(B) * unsigned(Hkv), kTopkThreads, 0, stream>>>(sel, scores, MBS, ctx,
                                                                               Hkv, BS, topk);
    return cudaGetLastError();
}

}  // namespace pa
