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
//    16-token KV block (dense: logical blocks 0..ceil(ctx/16)-1; sparse: the
//    topk selection entries); the E4M3 cache takes two consecutive blocks
//    (or entries) per item, so that its items carry the bytes of a bf16 one. The segments are concatenated and cut into
//    equal contiguous ranges, one per CTA of a persistent grid (one CTA per
//    SM), so every SM streams the same number of KV bytes whatever the
//    length mix.
//  * Data movement. A producer warp walks the CTA's range, resolves each
//    item's physical block (block table, and selection for sparse) a window
//    of 32 items ahead, and issues two TMA tile loads per K and per V block
//    ([16 tokens x 64 dims] boxes of a 4-D tensor map over the whole pool,
//    128-byte swizzle, L2 evict-first) into an S-stage shared-memory ring with
//    full/empty mbarriers. The physical block number is a runtime TMA
//    coordinate.
//    The producer's lanes work on 8 items at a time (one lane per tile copy),
//    so one warp instruction issues up to 32 TMA copies.
//  * Math. Consumer warps take the ring's items in pairs (E4M3: one
//    two-block item), round-robin; the ring's depth is a multiple of that
//    round so that every stage belongs to one consumer.
//    The GQA group's queries stay in registers as mma B fragments; S^T = K Q^T
//    and O^T += V^T P^T run on bf16 mma.sync (m16n8k16) with the tokens as M
//    and the (up to 8) heads of the group as N, so every K/V byte serves the
//    whole group. Online softmax in the log2 domain over 32 tokens per step
//    (running max, normaliser, accumulator rescaled only when the max grows);
//    P is rounded to bf16 and transposed in registers with movmatrix.
//  * Masking. Tokens past ctx get score -inf and their V fragment lanes are
//    zeroed, so NaN/Inf garbage in unused slots never reaches the output.
//  * Combine. At the end of each segment every consumer warp deposits its
//    state in shared memory and moves on; a merge warp (one query row per
//    sequence) merges the states, so a merge never holds a consumer's ring
//    stages and stalls the in-order producer. A CTA holding a whole segment
//    writes bf16 output; otherwise the merge warp writes a normalised
//    partial and its log2-sum-exp, and in the last CTA to arrive (atomic
//    counter per segment, reset to zero afterwards) merges the pieces with
//    weights exp2(lse_s - max lse).
#include "common.cuh"
#include "kernels.h"

namespace pa {

namespace {

// Launch geometry (tuning knobs): consumer warps, and item pairs (E4M3:
// two-block items) each consumer has in flight. The ring has S = 2 *
// consumers * pairs stages (E4M3: consumers * items), so stage s always
// belongs to consumer (s / 2) % consumers (E4M3: s % consumers): every
// consumer waits on its own stages in order and an mbarrier parity wait can
// never be answered by an older phase.
// Three consumers, the producer and the merge warp: five warps at 248
// registers each carry the HBM rate and leave room for the selection's CTAs
// beside a decode CTA. The multi-token kernel keeps one consumer per query
// row of a group (kMultiRowGroup) and no merge warp.
#ifndef PA_DECODE_CONSUMERS
#define PA_DECODE_CONSUMERS 3
#endif
#ifndef PA_DECODE_PAIRS
#define PA_DECODE_PAIRS 4
#endif
#ifndef PA_DECODE_PAIRS_MULTI
#define PA_DECODE_PAIRS_MULTI 3
#endif
// E4M3 cache: consumer warps and two-block items in flight per consumer. Six
// consumers, the producer and the merge warp are eight warps: two per
// register-file partition (a ninth warp would cap registers at 168 and
// spill).
#ifndef PA_DECODE_CONSUMERS_F8
#define PA_DECODE_CONSUMERS_F8 6
#endif
#ifndef PA_DECODE_PAIRS_F8
#define PA_DECODE_PAIRS_F8 3
#endif
// Registers per thread. With five warps, one register-file partition holds
// two decode warps; at 184 registers each (11,776 of the partition's 16,384)
// two warps of a selection kernel (64 registers each) still fit beside them,
// so the Quest path's scoring can run on the SMs the dense decode occupies.
// The kernel needs no spills at this cap (the combine loads two pieces per
// round).
#ifndef PA_DECODE_MAXNREG
#define PA_DECODE_MAXNREG 184
#endif

// Sparse decode of small selections (fewer than kSparseLargeItems items per
// SM): the grid follows the segments, pieces of at least kSparseMinItems items.
constexpr int kSparseMinItems = 16;

template <int D, bool F8 = false, bool MULTI = false>
struct DecodeCfg {
    static_assert(!F8 || D == 128, "the E4M3 cache path is for head_dim 128");
    static constexpr int BS = kBlockSize;
    static constexpr int KT = BS * D * (F8 ? 1 : 2);  // bytes of one K (or V) tile
    // KV blocks per item: the E4M3 cache takes two consecutive blocks of a
    // segment per item, so that an item moves as many bytes as a bf16 one
    // (the loop is bound per item at small items)
    static constexpr int BPI = F8 ? 2 : 1;
    static constexpr int STAGE = 2 * KT * BPI;  // K + V of the item's blocks
    static constexpr int NKK = D / 16;          // QK k-steps == PV m-tiles
    static constexpr int HALF = BS * 128;       // bytes of one 64-dim half tile
    static constexpr int PART = D * 8 + 8;      // floats per partial slot: O[D][8], lse[8]
    static constexpr int NC = F8 ? PA_DECODE_CONSUMERS_F8 : (MULTI ? kMultiRowGroup : PA_DECODE_CONSUMERS);
    // one query row per sequence: a merge warp after the producer takes the
    // segment-end merges off the consumers
    static constexpr int MW = MULTI ? 0 : 1;
    static constexpr int THREADS = (NC + 1 + MW) * 32;
    static constexpr int PAIRS = MULTI ? PA_DECODE_PAIRS_MULTI : PA_DECODE_PAIRS;
    static constexpr int R = F8 ? PA_DECODE_PAIRS_F8 : (D == 128 ? PAIRS : 2 * PAIRS);
    // stages per consumer step: bf16 takes items in pairs, E4M3 one (two-block) item
    static constexpr int SPS = F8 ? 1 : 2;
    static constexpr int S = SPS * NC * R;      // ring stages
    static constexpr int SCR = D * 8 + 16;      // floats per consumer merge slot: acc[D][8], m[8], l[8]
    static constexpr size_t off_bars = size_t(S) * STAGE;
    static constexpr size_t off_info = off_bars + size_t(S) * 16;
    // E4M3 cache: each stage's K and V scales (float4: the two blocks) after the item info
    static constexpr size_t off_iscale = off_info + size_t(S) * 8;
    static constexpr size_t off_scr = off_iscale + (F8 ? size_t(S) * 16 : 0);
    static constexpr size_t off_flags = off_scr + size_t(NC) * SCR * 4;
    static constexpr size_t off_pre = off_flags + 64;
    // per-row item prefix (PB + 1 entries); multi-token rows then add each
    // row group's sequence and first query row (R entries each)
    static constexpr size_t seq_off(int PB) { return off_pre + (size_t(PB + 1) * 4 + 15) / 16 * 16; }
    static constexpr size_t row0_off(int PB, int R) { return seq_off(PB) + (size_t(R) * 2 + 15) / 16 * 16; }
    static constexpr size_t smem_bytes(int PB, int R = 0) { return 1024 + row0_off(PB, R) + (size_t(R) * 2 + 15) / 16 * 16; }
    // fused Quest decode (one query row per sequence): the CTA's selection
    // entries [nsel] after the per-row prefix
    static constexpr size_t sel_off(int PB) { return row0_off(PB, 0); }
    static constexpr size_t smem_bytes_sel(int PB, int nsel) { return 1024 + sel_off(PB) + size_t(nsel) * 4; }
    // top-K scratch of the fused Quest decode, in the ring (free until the
    // first copy): the keys, then one 256-bin histogram per warp and the
    // per-warp counts
    static constexpr int TOPK_HC = THREADS / 32;
    static constexpr size_t TOPK_SCRATCH = size_t(TOPK_HC) * 1024 + 256;
    static constexpr int KEYS_CAP = int((size_t(S) * STAGE - TOPK_SCRATCH) / 4);
    static constexpr size_t off_topk_hist = size_t(S) * STAGE - TOPK_SCRATCH;
};

// One binary serves the dense call and the sparse one (topk > 0: the items
// are the selected blocks), so either call runs code the other has just
// brought into the SMs' instruction caches; code that runs once per CTA (the
// prologue, the merge and the combine) is otherwise fetched cold, several
// microseconds per launch.
// BSC (E4M3 cache only): per-block scales, read per item, instead of one K
// and V scale per KV head.
template <int D, bool F8, bool MULTI, bool BSC = false>
__global__ void __maxnreg__(PA_DECODE_MAXNREG)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const DecodeArgs a) {
    using C = DecodeCfg<D, F8, MULTI>;
    static_assert(!BSC || (F8 && !MULTI), "per-block scales: the E4M3 cache, one query row");
    constexpr bool PSC = F8 && BSC;  // per-item scales
    const bool SPARSE = !MULTI && a.topk > 0;
    constexpr int BS = C::BS, NC = C::NC, S = C::S, NKK = C::NKK, BPI = C::BPI;

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t base = (raw + 1023u) & ~1023u;
    uint8_t *bp = smem_raw + (base - raw);
    const uint32_t full_bar = base + uint32_t(C::off_bars);
    const uint32_t empty_bar = full_bar + S * 8;
    int2 *info = reinterpret_cast<int2 *>(bp + C::off_info);
    float4 *iscale = reinterpret_cast<float4 *>(bp + C::off_iscale);  // E4M3 cache only
    float *scr = reinterpret_cast<float *>(bp + C::off_scr);
    volatile int *flags = reinterpret_cast<volatile int *>(bp + C::off_flags);
    const uint32_t merge_bar = base + uint32_t(C::off_flags) + 16;  // consumers' deposits (count NC)
    int32_t *pre = reinterpret_cast<int32_t *>(bp + C::off_pre);
    // multi-token rows: a work-list row is a group of up to RG query rows of
    // one sequence; seq_of / row0_of give its sequence and first query row
    constexpr int RG = C::NC;
    static_assert(!MULTI || RG == kMultiRowGroup, "multi-token rows: one query row per consumer warp");
    const int PB = MULTI ? max(a.B, a.nseq) : a.B;
    uint16_t *seq_of = reinterpret_cast<uint16_t *>(bp + C::seq_off(PB));
    uint16_t *row0_of = reinterpret_cast<uint16_t *>(bp + C::row0_off(PB, a.B));

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B, Hkv = a.Hkv, G = a.G;
    const int max_tok = a.MBS * BS;

    // ---- prologue: items per KV head of every sequence and their prefix sum
    pdl_trigger();
    if (tid == 0) {
        prefetch_tensormap(&tm_k);
        prefetch_tensormap(&tm_v);
    }
    {
        // While the previous kernel finishes: pull this CTA's share of the
        // context lengths, block table and selection into L2 (hints only).
        const int64_t nthr = int64_t(gridDim.x) * C::THREADS;
        const int64_t gt = int64_t(blockIdx.x) * C::THREADS + tid;
        const int nseq = MULTI ? a.nseq : B;  // ctx and block tables are per sequence
        for (int64_t off = gt * 32; off < int64_t(nseq); off += nthr * 32) prefetch_l2(a.ctx + off);
        const int64_t bt_n = int64_t(nseq) * a.MBS;
        for (int64_t off = gt * 32; off < bt_n; off += nthr * 32) prefetch_l2(a.bt + off);
        if (SPARSE && !a.scores) {
            const int64_t sel_n = int64_t(B) * Hkv * a.topk;
            for (int64_t off = gt * 32; off < sel_n; off += nthr * 32) prefetch_l2(a.sel + off);
        }
    }
    // Every call builds its per-sequence prefix from the context lengths (and
    // the query-row offsets of multi-token rows) while the previous kernel in
    // the stream finishes: the caller's inputs, which no kernel of this
    // library writes. The bf16 dense call also reads only block-table entries
    // before its first copy, so its producer resolves its first items too and
    // waits for that kernel just before issuing copies; its consumers wait
    // before they touch q, the outputs or the workspace. Every other call
    // waits once the prefix is built.
    const bool early = !MULTI && !F8 && !SPARSE;
    // Multi-token rows ("18 e2e inference serving", sections 2.7 and 3.3):
    // query row r of sequence s (cu_q[s] <= r < cu_q[s+1]) sees the
    // positions before ctx_s - q_len_s + (r - cu_q[s]) + 1 (causal mask
    // aligned on the right).
    auto row_ctx = [&](int r, int s) -> int {
        const int c0 = min(max(__ldg(a.ctx + s), 0), max_tok);
        const int c1 = __ldg(a.cu_q + s), ql = __ldg(a.cu_q + s + 1) - c1;
        return min(max(c0 - ql + (r - c1) + 1, 0), c0);
    };
    // block count of work-list row v (MULTI: the blocks its last query row sees)
    auto row_items = [&](int v) -> int {
        int c;
        if constexpr (MULTI) {
            const int sq = seq_of[v];
            c = row_ctx(min(int(row0_of[v]) + RG, __ldg(a.cu_q + sq + 1)) - 1, sq);
        } else {
            c = min(max(__ldg(a.ctx + v), 0), max_tok);
        }
        const int nblk = (c + BS - 1) / BS;
        return SPARSE ? (nblk > 0 ? (a.topk + BPI - 1) / BPI : 0) : (nblk + BPI - 1) / BPI;
    };
    auto scan_pre = [&](int n) {  // pre[1..n] -> inclusive prefix sums (warp 0)
        if (warp == 0) {
            int carry = 0;
            for (int b0 = 0; b0 < n; b0 += 32) {
                const int b = b0 + lane;
                int v = (b < n) ? pre[b + 1] : 0;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int u = __shfl_up_sync(0xffffffffu, v, o);
                    if (lane >= o) v += u;
                }
                if (b < n) pre[b + 1] = carry + v;
                carry += __shfl_sync(0xffffffffu, v, 31);
            }
        }
    };
    if (tid == 0) {
        pre[0] = 0;
        flags[0] = 0;  // abort
        flags[2] = 0;  // segment ends whose states the merge warp has read
        for (int s = 0; s < S; ++s) {
            mbar_init(full_bar + s * 8, 1);
            mbar_init(empty_bar + s * 8, MULTI ? NC : 1);  // MULTI: every consumer reads every stage
        }
        if (!MULTI) mbar_init(merge_bar, NC);
        fence_barrier_init();
    }
    int NR = B;  // work-list rows
    if constexpr (MULTI) {
        // row groups: ceil(q_len / RG) per sequence, then each group's sequence and first row
        for (int sq = tid; sq < a.nseq; sq += C::THREADS) {
            const int ql = max(__ldg(a.cu_q + sq + 1) - __ldg(a.cu_q + sq), 0);
            pre[sq + 1] = (ql + RG - 1) / RG;
        }
        __syncthreads();
        scan_pre(a.nseq);
        __syncthreads();
        NR = min(pre[a.nseq], B);
        for (int sq = tid; sq < a.nseq; sq += C::THREADS) {
            const int g0 = pre[sq], r0 = __ldg(a.cu_q + sq);
            for (int gi = g0; gi < min(pre[sq + 1], NR); ++gi) {
                seq_of[gi] = uint16_t(sq);
                row0_of[gi] = uint16_t(min(r0 + (gi - g0) * RG, 0xffff));
            }
        }
        __syncthreads();
    }
    if constexpr (MULTI) {
        for (int v = tid; v < NR; v += C::THREADS) pre[v + 1] = row_items(v);
    } else {
        // eight independent context-length loads per thread in flight
        for (int v0 = tid; v0 < NR; v0 += 8 * C::THREADS) {
            int c8[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * C::THREADS;
                c8[u] = v < NR ? __ldg(a.ctx + v) : 0;
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = v0 + u * C::THREADS;
                if (v < NR) {
                    const int nblk = (min(max(c8[u], 0), max_tok) + BS - 1) / BS;
                    pre[v + 1] = SPARSE ? (nblk > 0 ? (a.topk + BPI - 1) / BPI : 0) : (nblk + BPI - 1) / BPI;
                }
            }
        }
    }
    __syncthreads();
    scan_pre(NR);
    __syncthreads();
    if (!early) pdl_wait();  // the rest may read what the previous kernel wrote

    // sequences (MULTI: query rows of groups) with nothing to attend to get a zero output
    if constexpr (MULTI) {
        for (int idx = blockIdx.x * C::THREADS + tid; idx < NR * RG * a.Hq; idx += gridDim.x * C::THREADS) {
            const int v = idx / (RG * a.Hq), r = (idx / a.Hq) % RG, h = idx % a.Hq;
            const int row = row0_of[v] + r;
            if (pre[v + 1] == pre[v] && row < __ldg(a.cu_q + seq_of[v] + 1) && row < B) {
                uint4 *o = reinterpret_cast<uint4 *>(a.out + (int64_t(row) * a.Hq + h) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
            }
        }
    } else if (!early || warp < NC) {  // early: the consumers, after their wait
        if (early) pdl_wait();
        const int nt = early ? NC * 32 : C::THREADS;
        for (int idx = blockIdx.x * nt + tid; idx < B * a.Hq; idx += gridDim.x * nt) {
            const int b = idx / a.Hq;
            if (pre[b + 1] == pre[b]) {
                uint4 *o = reinterpret_cast<uint4 *>(a.out + int64_t(idx) * D);
#pragma unroll
                for (int i = 0; i < D / 8; ++i) o[i] = make_uint4(0, 0, 0, 0);
            }
        }
        if (SPARSE && a.scores)  // fused Quest decode: sequences with no blocks select nothing
            for (int64_t idx = int64_t(blockIdx.x) * C::THREADS + tid; idx < int64_t(B) * Hkv * a.topk;
                 idx += int64_t(gridDim.x) * C::THREADS) {
                const int b = int(idx / (int64_t(Hkv) * a.topk));
                if (pre[b + 1] == pre[b]) a.sel_out[idx] = -1;
            }
    }

    const int64_t total = int64_t(Hkv) * pre[NR];
    const int64_t L = (total + gridDim.x - 1) / gridDim.x;
    const int64_t pos0 = int64_t(blockIdx.x) * L;
    const int64_t pos1 = min(total, pos0 + L);
    if (pos0 >= pos1) return;  // whole CTA: nothing to do
    const int n_items = int(pos1 - pos0);

    // sequence holding global item position p
    auto find_seq = [&](int64_t p) -> int {
        int lo = 0, hi = NR;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (int64_t(Hkv) * pre[mid] <= p) lo = mid; else hi = mid;
        }
        return lo;
    };

    // ---- fused Quest decode: this CTA selects, for every segment it holds a
    // piece of, the top-K blocks of that (sequence, KV head) from the scores
    // ([P1] "Quest Sparse Attention": ties to the lower block index), keeps
    // its piece of the selection in shared memory, and the CTA holding the
    // segment's first entry writes the selection row out. The same rule as
    // quest_select_topk (cta_topk_threshold / cta_topk_emit).
    int32_t *sel_s = reinterpret_cast<int32_t *>(bp + C::sel_off(PB));
    if (SPARSE && a.scores) {
        uint32_t *keys = reinterpret_cast<uint32_t *>(bp);  // the ring: no copy has been issued yet
        int *hist = reinterpret_cast<int *>(bp + C::off_topk_hist);
        int *wcnt = hist + C::TOPK_HC * 256;  // scratch of the top-K helpers
        int64_t p = pos0;
        int b = find_seq(p);
        int kvh = int((p - int64_t(Hkv) * pre[b]) / (pre[b + 1] - pre[b]));
        while (p < pos1) {
            const int nseg = pre[b + 1] - pre[b];
            const int seg = b * Hkv + kvh;
            const int64_t s0 = int64_t(Hkv) * pre[b] + int64_t(kvh) * nseg;
            const int64_t e0 = s0 + nseg;
            // this CTA's entries [i0, i1) (BPI per item): entry r -> mine[r]
            const int i0 = BPI * int(p - s0), i1 = BPI * int(min(e0, pos1) - s0);
            int32_t *mine = sel_s + BPI * (p - pos0) - i0;
            const bool writer = s0 >= pos0;                            // holds entry 0: writes the row
            int32_t *orow = a.sel_out + int64_t(seg) * a.topk;
            const float *srow = a.scores + int64_t(seg) * a.MBS;
            const int n = (min(max(__ldg(a.ctx + b), 0), max_tok) + BS - 1) / BS;
            const int topk = a.topk;
            if (n <= topk) {
                for (int i = tid; i < topk; i += C::THREADS) {
                    const int v = i < n ? i : -1;
                    if (writer) orow[i] = v;
                    if (i >= i0 && i < i1) mine[i] = v;
                }
            } else {
                const bool cached = n <= C::KEYS_CAP;
                if (cached) cta_load_keys<C::THREADS>(keys, srow, n);
                auto key_of = [&](int j) -> uint32_t { return cached ? keys[j] : f32_order_key(__ldcg(srow + j)); };
                uint32_t thr;
                int keq;
                cta_topk_threshold<C::THREADS, C::TOPK_HC>(key_of, n, topk, hist, wcnt, thr, keq);
                cta_topk_emit<C::THREADS>(key_of, n, thr, keq, wcnt, [&](int r, int j) {
                    if (writer) orow[r] = j;
                    if (r >= i0 && r < i1) mine[r] = j;
                });
            }
            __syncthreads();  // keys and counts are reused by the next segment
            p = min(e0, pos1);
            if (++kvh == Hkv) {
                kvh = 0;
                do {
                    ++b;
                } while (b < NR && pre[b + 1] == pre[b]);
            }
        }
    }

    if (warp == NC) {
        // ================================================================ producer
        // Item windows of 32 (one item per lane), refilled in three steps so no
        // load is waited on before its value is needed: stage C locates the
        // item and starts loading ctx (and the selection entry for sparse);
        // one window later stage B starts loading the block-table entry; one
        // window after that the items are issued.
        // an item's logical blocks j, j1 (j1: the second block of an E4M3
        // item, -1 if none), their physical blocks and their K and V scales
        struct Win {
            int seg, j, phys, ctxv;
            float sk, sv;  // E4M3 cache: the item's K and V scale
            int j1, phys1;
            float sk1, sv1;
        };
        const Win none{-1, -1, -1, 0, 0.f, 0.f, -1, -1, 0.f, 0.f};
        auto stage_c = [&](int k0) -> Win {
            Win it = none;
            const int k = k0 + lane;
            if (k >= n_items) return it;
            const int64_t p = pos0 + k;
            const int b = find_seq(p);
            const int n = pre[b + 1] - pre[b];
            const int64_t r = p - int64_t(Hkv) * pre[b];
            const int kvh = int(r / n);
            const int i = int(r - int64_t(kvh) * n);
            it.seg = b * Hkv + kvh;
            if constexpr (MULTI) {
                const int sq = seq_of[b];
                it.ctxv = row_ctx(min(int(row0_of[b]) + RG, __ldg(a.cu_q + sq + 1)) - 1, sq);
            } else {
                it.ctxv = __ldg(a.ctx + b);
            }
            if constexpr (BPI == 1) {
                it.j = !SPARSE ? i : a.scores ? sel_s[k] : __ldg(a.sel + (int64_t(b) * Hkv + kvh) * a.topk + i);
            } else {  // entries e, e + 1 of the segment (blocks for dense, selection entries for sparse)
                const int e = BPI * i;
                const int32_t *srow = a.sel + (int64_t(b) * Hkv + kvh) * a.topk;
                if (!SPARSE) {
                    it.j = e;
                    it.j1 = e + 1;
                } else if (a.scores) {
                    it.j = sel_s[BPI * k];
                    it.j1 = e + 1 < a.topk ? sel_s[BPI * k + 1] : -1;
                } else {
                    it.j = __ldg(srow + e);
                    it.j1 = e + 1 < a.topk ? __ldg(srow + e + 1) : -1;
                }
            }
            return it;
        };
        auto stage_b = [&](Win &it) {
            if (it.seg < 0) return;
            const int b = it.seg / Hkv;
            const int s = MULTI ? int(seq_of[b]) : b;  // the row's sequence
            it.phys = (it.j >= 0 && it.j < a.MBS) ? __ldg(a.bt + int64_t(s) * a.MBS + it.j) : -1;
            if (BPI > 1) it.phys1 = (it.j1 >= 0 && it.j1 < a.MBS) ? __ldg(a.bt + int64_t(s) * a.MBS + it.j1) : -1;
        };
        // per-block scales: the item's K and V scale of its (physical block,
        // KV head); the load depends on the block-table entry, so it runs one
        // window after stage B
        auto stage_s = [&](Win &it) {
            if constexpr (PSC) {
                if (it.seg < 0) return;
                if (it.phys1 >= 0 && int64_t(it.phys1) < a.NB) {
                    const int64_t si = int64_t(it.phys1) * Hkv + it.seg % Hkv;
                    it.sk1 = __ldg(a.k_scale + si);
                    it.sv1 = __ldg(a.v_scale + si);
                }
                if (it.phys < 0 || int64_t(it.phys) >= a.NB) return;
                const int64_t si = int64_t(it.phys) * Hkv + it.seg % Hkv;
                it.sk = __ldg(a.k_scale + si);
                it.sv = __ldg(a.v_scale + si);
            }
        };
        // dense decode with the step's write: sequence seg / Hkv's new token,
        // KV head seg % Hkv, into physical block ph_w at offset (c_w - 1) % BS
        // (when the token's slot is that one), by the whole warp: lanes
        // [0, D/8) copy 16 bytes of K each and merge the metadata, lanes
        // [D/8, D/4) copy V
        auto write_new_token = [&](int seg_w, int ph_w, int c_w) {
            if constexpr (!F8 && !MULTI) {
                const int b = seg_w / Hkv, kvh = seg_w % Hkv, o = (c_w - 1) % BS;
                constexpr int VPR = D / 8;  // 16-byte vectors per KV-head row
                const int half = lane / VPR, e = lane % VPR;
                const bool meta = half == 0 && a.kmin_w && o != 0;
                const int64_t mrow = (int64_t(ph_w) * Hkv + kvh) * D;
                uint4 *mn = a.kmin_w ? reinterpret_cast<uint4 *>(a.kmin_w + mrow) + e : nullptr;
                uint4 *mx = a.kmin_w ? reinterpret_cast<uint4 *>(a.kmax_w + mrow) + e : nullptr;
                // every load in flight before the first use: the slot, the
                // token's 16 bytes, the block's metadata
                const int64_t slot = __ldg(a.new_slots + b);
                uint4 x = make_uint4(0u, 0u, 0u, 0u), lo = x, hi = x;
                if (half < 2)
                    x = __ldg(reinterpret_cast<const uint4 *>((half ? a.new_v : a.new_k) + (int64_t(b) * Hkv + kvh) * D) +
                              e);
                if (meta) {
                    lo = *mn;
                    hi = *mx;
                }
                if (slot != int64_t(ph_w) * BS + o || half >= 2) return;
                reinterpret_cast<uint4 *>((half ? a.vc_w : a.kc_w) + ((int64_t(ph_w) * BS + o) * Hkv + kvh) * D)[e] = x;
                if (half == 0 && a.kmin_w) {  // reset at offset 0, else merge
                    if (meta) {
                        minmax_bf16x2(lo.x, hi.x, x.x);
                        minmax_bf16x2(lo.y, hi.y, x.y);
                        minmax_bf16x2(lo.z, hi.z, x.z);
                        minmax_bf16x2(lo.w, hi.w, x.w);
                    } else {
                        lo = x;
                        hi = x;
                    }
                    *mn = lo;
                    *mx = hi;
                }
            }
        };
        const uint64_t policy = l2_policy_evict_first();
        if (SPARSE && a.scores) fence_proxy_async();  // the ring held the top-K scratch
        Win wa = stage_c(0), wb = stage_c(32);
        stage_b(wa);
        stage_b(wb);
        Win wc = stage_c(64);
        // per-block scales: a fourth window, so the scale loads (stage S) have
        // a window to land in: wa issued, wb scales, wc block-table entries,
        // wd context and selection
        Win wd = none;
        if constexpr (PSC) {
            stage_b(wc);
            wd = stage_c(96);
            stage_s(wa);
            stage_s(wb);
        }
        if (early) pdl_wait();  // the first items are resolved: now the previous kernel
        int wbase = 0;
        int issued = 0;  // items [0, issued) have been armed
        int fail_step = 0;
        unsigned fail_armed = 0;  // after a failure: leader lanes whose item was armed
        // IPS items per step, LPI lanes per item: lane = LPI * item + part,
        // part = which tile copy (bf16: K and V in two 64-dim halves each;
        // E4M3: K and V of each of the item's two blocks)
        constexpr int LPI = 4, IPS = 32 / LPI;
        // a step's items take distinct stages, and each waits only for items
        // of earlier steps to leave its stage (no two items of a step alias)
        static_assert(IPS < S, "items per producer step must stay below the ring depth");
        const int it = lane / LPI, part = lane % LPI;
        constexpr int PARTS = F8 ? 2 * BPI : 2 * (D / 64);  // K and V (bf16: 64-dim halves)
        for (int k0 = 0; k0 < n_items; k0 += IPS) {
            if (k0 >= a.stop_item) break;  // failure tests: the stages from here on are never armed
            if (k0 >= wbase + 32) {
                wa = wb;
                wb = wc;
                if constexpr (PSC) {
                    wc = wd;
                    stage_s(wb);
                    stage_b(wc);
                    wbase += 32;
                    wd = stage_c(wbase + 96);
                } else {
                    stage_b(wb);
                    wbase += 32;
                    wc = stage_c(wbase + 64);
                }
            }
            const int k = k0 + it;
            const int seg = __shfl_sync(0xffffffffu, wa.seg, k & 31);
            const int j = __shfl_sync(0xffffffffu, wa.j, k & 31);
            const int ph = __shfl_sync(0xffffffffu, wa.phys, k & 31);
            const int cv = __shfl_sync(0xffffffffu, wa.ctxv, k & 31);
            float sk = 0.f, sv = 0.f, sk1 = 0.f, sv1 = 0.f;
            if constexpr (PSC) {
                sk = __shfl_sync(0xffffffffu, wa.sk, k & 31);
                sv = __shfl_sync(0xffffffffu, wa.sv, k & 31);
                sk1 = __shfl_sync(0xffffffffu, wa.sk1, k & 31);
                sv1 = __shfl_sync(0xffffffffu, wa.sv1, k & 31);
            }
            const bool live = k < n_items;
            const int c = min(max(cv, 0), max_tok);
            const int nblk = (c + BS - 1) / BS;
            const bool valid = live && j >= 0 && j < nblk && ph >= 0 && int64_t(ph) < a.NB;
            const int nv = valid ? min(BS, c - j * BS) : 0;
            // E4M3: the item's second block (valid tokens nv1; info packs nv + nv1 * 256)
            int ph1 = -1, nv1 = 0;
            if constexpr (BPI > 1) {
                const int j1 = __shfl_sync(0xffffffffu, wa.j1, k & 31);
                ph1 = __shfl_sync(0xffffffffu, wa.phys1, k & 31);
                const bool valid1 = live && j1 >= 0 && j1 < nblk && ph1 >= 0 && int64_t(ph1) < a.NB;
                nv1 = valid1 ? min(BS, c - j1 * BS) : 0;
            }
            const int st = k % S;
            const uint32_t fb = full_bar + st * 8;
            // the item's leader lane waits for its stage to be released, then arms it
            int ok = 1;
            if (live && part == 0) {
                if (k >= S && !mbar_wait_bounded(empty_bar + st * 8, ((k / S) & 1) ^ 1, a.wait_ns)) {
                    ok = 0;
                } else {
                    info[st] = make_int2(MULTI ? j : seg, nv + (nv1 << 8));  // MULTI: consumers mask per query row
                    if constexpr (PSC) iscale[st] = make_float4(sk, sv, sk1, sv1);
                    const uint32_t bytes = BPI > 1 ? (nv > 0 ? 2u * C::KT : 0u) + (nv1 > 0 ? 2u * C::KT : 0u)
                                                   : (nv > 0 ? uint32_t(C::STAGE) : 0u);
                    if (bytes > 0) mbar_arrive_expect_tx(fb, bytes);
                    else mbar_arrive(fb);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, lane - part);
            __syncwarp();
            if constexpr (!F8 && !MULTI) {
                // with the step's write: a segment's last block gets the
                // sequence's new token before its copy is issued (this CTA is
                // the only reader of that block in the call)
                if (!SPARSE && a.new_k) {
                    unsigned wm = __ballot_sync(0xffffffffu, part == 0 && live && ok && nv > 0 && j == nblk - 1);
                    if (wm) {
                        while (wm) {
                            const int src = __ffs(wm) - 1;
                            wm &= wm - 1;
                            write_new_token(__shfl_sync(0xffffffffu, seg, src), __shfl_sync(0xffffffffu, ph, src),
                                            __shfl_sync(0xffffffffu, c, src));
                        }
                        fence_proxy_async_global();  // the copies below read what was written
                        __syncwarp();
                    }
                }
            }
            if constexpr (F8) {
                // parts: K and V of block 0, then of block 1. K: one [16 tokens
                // x 128 dims] byte box (tensor map); V: the block's [128 dims x
                // 16 tokens] byte matrix of this KV head, 2 KB of contiguous
                // bytes: one plain bulk copy
                const int blk = part >> 1;
                const int phb = blk ? ph1 : ph;
                if (live && ok && part < PARTS && (blk ? nv1 : nv) > 0) {
                    const uint32_t dst = base + st * C::STAGE + part * C::KT;
                    if ((part & 1) == 0) {
                        tma_load_4d(dst, &tm_k, fb, 0, seg % Hkv, 0, phb, policy);
                    } else {
                        const uint8_t *src = a.v8 + (int64_t(phb) * Hkv + seg % Hkv) * int64_t(C::KT);
                        bulk_load_1d(dst, src, uint32_t(C::KT), fb, policy);
                    }
                }
            } else if (live && ok && nv > 0 && part < PARTS) {
                constexpr int HV = D / 64;                   // 64-dim halves per tile
                const int tsel = part / HV, hf = part % HV;  // 0: K, 1: V
                const uint32_t dst = base + st * C::STAGE + tsel * C::KT + hf * C::HALF;
                tma_load_4d(dst, tsel ? &tm_v : &tm_k, fb, hf * 64, seg % Hkv, 0, ph, policy);
            }
            if (!__all_sync(0xffffffffu, ok)) {
                // a stage was never released: give up (consumers skip their
                // waits from now on), remembering which items of this step
                // were armed so their copies can land before the CTA exits
                if (lane == 0) {
                    flags[0] = 1;
                    atomicOr(a.status, kStatusTimeout);
                }
                fail_step = k0;
                fail_armed = __ballot_sync(0xffffffffu, live && part == 0 && ok);
                break;
            }
            issued = min(n_items, k0 + IPS);
        }
        // keep the CTA alive until every copy issued has landed (consumers that
        // gave up do not wait for them)
        if (lane == 0) {
            for (int k = max(0, issued - S); k < issued; ++k)
                mbar_wait_bounded(full_bar + (k % S) * 8, (k / S) & 1, a.wait_ns);
            for (int i = 0; i < IPS; ++i)
                if (fail_armed & (1u << (LPI * i))) {
                    const int k = fail_step + i;
                    mbar_wait_bounded(full_bar + (k % S) * 8, (k / S) & 1, a.wait_ns);
                }
        }
        return;
    }

    // ==================================================================== consumers
    const int c_id = warp;  // 0 .. NC-1
    const int g = lane >> 2, q4 = lane & 3;
    // E4M3 cache: times the segment's K scale (per-KV-head scales)
    float scale_log2 = a.scale_log2;
    // E4M3 cache: acc holds O / vref. Per-KV-head scales: vref is the
    // segment's V scale; per-block scales: the largest V scale of the
    // segment's blocks seen so far (0 before the first).
    float vref = 0.f;
    uint32_t qb[NKK][2];
    float acc[NKK][4];
    float m0, m1, l0, l1;

    // reset the running state and load query row qr's group of heads for
    // segment seg's KV head (qr < 0: zero queries)
    auto load_q = [&](int seg, int qr) {
        const int kvh = seg % Hkv;
        const int b = qr < 0 ? 0 : qr;
        const bool hv = g < G && qr >= 0;
        const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
            a.q + (int64_t(b) * a.Hq + kvh * G + (hv ? g : 0)) * D);
        if constexpr (F8) {
            // f16 B fragments in the k order the E4M3 K fragments come in:
            // k-step kk covers dims 16kk + 4*q4 + {0, 1} (b0) and {2, 3} (b1)
#pragma unroll
            for (int kk = 0; kk < NKK; ++kk) {
                const uint2 v = hv ? __ldg(reinterpret_cast<const uint2 *>(qrow + 8 * kk + 2 * q4))
                                   : make_uint2(0u, 0u);
                qb[kk][0] = pack_f16x2(bf16_lo(v.x), bf16_hi(v.x));
                qb[kk][1] = pack_f16x2(bf16_lo(v.y), bf16_hi(v.y));
            }
            if constexpr (BSC) {
                vref = 0.f;
            } else {
                scale_log2 = a.scale_log2 * __ldg(a.k_scale + kvh);
                vref = __ldg(a.v_scale + kvh);
            }
        } else {
#pragma unroll
            for (int kk = 0; kk < NKK; ++kk) {
                qb[kk][0] = hv ? __ldg(qrow + 8 * kk + q4) : 0u;
                qb[kk][1] = hv ? __ldg(qrow + 8 * kk + 4 + q4) : 0u;
            }
        }
#pragma unroll
        for (int mt = 0; mt < NKK; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
        m0 = m1 = -INFINITY;
        l0 = l1 = 0.f;
    };
    // S^T = K Q^T for the 16 tokens of one staged block (two mma chains)
    auto qk = [&](uint32_t kb, float (&sc)[4]) {
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
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = sa[e] + sb[e];
    };
    // O^T += V^T P^T for one staged block; V lanes of tokens >= nv zeroed
    auto pv = [&](uint32_t vb, uint32_t p01, uint32_t p23, int nv) {
        const uint32_t pb0 = movmatrix_trans(p01), pb1 = movmatrix_trans(p23);
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
    };
    // E4M3 tiles: one [16 tokens x 128 dims] byte box, 128-byte swizzle. An
    // ldmatrix.x4 of 16-bit pairs gives lane (g, q4) the 4 codes at dims
    // 32c + 4q4 .. +3 (and 32c + 16 + 4q4 ..) of tokens g and g + 8. For
    // S^T = K Q^T those are the A fragments of two k-steps with k = 2q4 + e
    // standing for dim 4q4 + e and k = 2q4 + 8 + e for dim 4q4 + 2 + e (the
    // query fragments use the same order); each code pair becomes an f16 pair.
    auto qk8 = [&](uint32_t kb, float (&sc)[4]) {
        float sa[4] = {0.f, 0.f, 0.f, 0.f}, sb[4] = {0.f, 0.f, 0.f, 0.f};
        const int rk = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
        for (int c2 = 0; c2 < NKK / 2; ++c2) {
            const int ch = 2 * c2 + (lane >> 4);
            uint32_t r0, r1, r2, r3;
            ldsm_x4(kb + rk * 128 + ((ch ^ (lane & 7)) << 4), r0, r1, r2, r3);
            uint32_t h0l, h0h, h1l, h1h, h2l, h2h, h3l, h3h;
            e4m3x4_to_f16x2x2(r0, h0l, h0h);
            e4m3x4_to_f16x2x2(r1, h1l, h1h);
            e4m3x4_to_f16x2x2(r2, h2l, h2h);
            e4m3x4_to_f16x2x2(r3, h3l, h3h);
            mma_f16(sa, h0l, h1l, h0h, h1h, qb[2 * c2][0], qb[2 * c2][1]);
            mma_f16(sb, h2l, h3l, h2h, h3h, qb[2 * c2 + 1][0], qb[2 * c2 + 1][1]);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = sa[e] + sb[e];
    };
    // O^T += V^T P^T from an E4M3 V tile, stored per block and KV head as a
    // [128 dims x 16 tokens] byte matrix with the tokens of a row in the
    // order 0 1 8 9 2 3 10 11 ...: an ldmatrix.x4 over 32 consecutive dim
    // rows gives lane (g, q4) the codes of tokens 2q4, 2q4+1, 8+2q4, 9+2q4 of
    // dims g, g+8, g+16, g+24 -- after conversion exactly the V^T A
    // fragments of two m-tiles (rows = dims, k = tokens), no transpose.
    auto pv8 = [&](uint32_t vb, uint32_t p01, uint32_t p23, int nv) {
        const uint32_t pb0 = movmatrix_trans(p01), pb1 = movmatrix_trans(p23);
        const bool part_blk = nv < BS;
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (part_blk) {
            const int t0 = 2 * q4;
            mlo = (t0 < nv ? 0x0000ffffu : 0u) | (t0 + 1 < nv ? 0xffff0000u : 0u);
            mhi = (t0 + 8 < nv ? 0x0000ffffu : 0u) | (t0 + 9 < nv ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int c2 = 0; c2 < NKK / 2; ++c2) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4(vb + (32 * c2 + lane) * 16, r0, r1, r2, r3);
            uint32_t a0, a2, a1, a3, b0, b2, b1, b3;
            e4m3x4_to_f16x2x2(r0, a0, a2);
            e4m3x4_to_f16x2x2(r1, a1, a3);
            e4m3x4_to_f16x2x2(r2, b0, b2);
            e4m3x4_to_f16x2x2(r3, b1, b3);
            if (part_blk) {  // tokens past the context: zero V (garbage may be NaN)
                a0 &= mlo; a1 &= mlo; a2 &= mhi; a3 &= mhi;
                b0 &= mlo; b1 &= mlo; b2 &= mhi; b3 &= mhi;
            }
            mma_f16(acc[2 * c2], a0, a1, a2, a3, pb0, pb1);
            mma_f16(acc[2 * c2 + 1], b0, b1, b2, b3, pb0, pb1);
        }
    };
    // wait for an item's stage (skipped once the CTA has given up); returns
    // the item's valid token count
    auto wait_full = [&](int k) -> int {
        if (flags[0]) return 0;
        if (!mbar_wait_bounded(full_bar + (k % S) * 8, (k / S) & 1, a.wait_ns)) {
            if (lane == 0) {
                flags[0] = 1;
                atomicOr(a.status, kStatusTimeout);
            }
            return 0;
        }
        return info[k % S].y;
    };
    // MULTI: the item's logical block too (each consumer masks its own row)
    auto wait_full_j = [&](int k, int &j) -> int {
        const int nv = wait_full(k);
        j = info[k % S].x;
        return nv;
    };
    // one online-softmax step over up to two staged blocks at shared-memory
    // addresses s0a, s1a (K tile, then V tile; nv == 0: no block), with their
    // K and V scales ca, cb (per-block scales only)
    auto step = [&](uint32_t s0a, int nva, float2 ca, uint32_t s1a, int nvb, float2 cb) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        float sla = scale_log2, slb = scale_log2;  // per-block scales: times the blocks' K scales
        float ra = 1.f, rb = 1.f, vr = 1.f;        // per-block scales: V scale ratios, warp-uniform
        if constexpr (F8) {
            if (nva > 0) qk8(s0a, s0);
            if (nvb > 0) qk8(s1a, s1);
        } else {
            if (nva > 0) qk(s0a, s0);
            if (nvb > 0) qk(s1a, s1);
        }
        if constexpr (PSC) {
            // Each block's V codes stand for decode(code) * sv. acc is kept in
            // units of vref = the largest sv so far: a block with a larger sv
            // rescales acc by vref / sv first; a block's P enters the PV
            // product times sv / vref (a power of two, so the f16 product is
            // exact down to the f16 subnormal range).
            sla = scale_log2 * ca.x;
            slb = scale_log2 * cb.x;
            float vnew = vref;
            if (nva > 0) vnew = fmaxf(vnew, ca.y);
            if (nvb > 0) vnew = fmaxf(vnew, cb.y);
            // the ratios are exact: the scales are powers of two between
            // 2^-126 and 2^120 (the largest bf16 value over 448), so dividing
            // by vnew is a product with its exact reciprocal
            const float rv = rcp_pow2(vnew);
            if (vnew != vref) {
                vr = vref * rv;
                vref = vnew;
            }
            if (nva > 0 && ca.y != vnew) ra = ca.y * rv;
            if (nvb > 0 && cb.y != vnew) rb = cb.y * rv;
        }
        const float x0 = (g < nva) ? s0[0] * sla : -INFINITY;
        const float x1 = (g < nva) ? s0[1] * sla : -INFINITY;
        const float x2 = (g + 8 < nva) ? s0[2] * sla : -INFINITY;
        const float x3 = (g + 8 < nva) ? s0[3] * sla : -INFINITY;
        const float y0 = (g < nvb) ? s1[0] * slb : -INFINITY;
        const float y1 = (g < nvb) ? s1[1] * slb : -INFINITY;
        const float y2 = (g + 8 < nvb) ? s1[2] * slb : -INFINITY;
        const float y3 = (g + 8 < nvb) ? s1[3] * slb : -INFINITY;
        float bm0 = fmaxf(fmaxf(x0, x2), fmaxf(y0, y2));
        float bm1 = fmaxf(fmaxf(x1, x3), fmaxf(y1, y3));
#pragma unroll
        for (int o = 4; o < 32; o <<= 1) {
            bm0 = fmaxf(bm0, __shfl_xor_sync(0xffffffffu, bm0, o));
            bm1 = fmaxf(bm1, __shfl_xor_sync(0xffffffffu, bm1, o));
        }
        const float mn0 = fmaxf(m0, bm0), mn1 = fmaxf(m1, bm1);
        const float r0 = (mn0 == -INFINITY) ? 0.f : mn0;
        const float r1 = (mn1 == -INFINITY) ? 0.f : mn1;
        const bool grow = (mn0 != m0) || (mn1 != m1);
        float al0 = fast_exp2(m0 - r0), al1 = fast_exp2(m1 - r1);
        // P rounded to the mma input type (bf16, or f16 for an E4M3 cache);
        // the normaliser sums the rounded values
        auto pk = [](float lo, float hi) { return F8 ? pack_f16x2(lo, hi) : pack_bf16x2(lo, hi); };
        auto plo = [](uint32_t v) { return F8 ? f16_lo(v) : bf16_lo(v); };
        auto phi = [](uint32_t v) { return F8 ? f16_hi(v) : bf16_hi(v); };
        const uint32_t p01 = pk(fast_exp2(x0 - r0), fast_exp2(x1 - r1));
        const uint32_t p23 = pk(fast_exp2(x2 - r0), fast_exp2(x3 - r1));
        const uint32_t q01 = pk(fast_exp2(y0 - r0), fast_exp2(y1 - r1));
        const uint32_t q23 = pk(fast_exp2(y2 - r0), fast_exp2(y3 - r1));
        l0 = l0 * al0 + ((plo(p01) + plo(p23)) + (plo(q01) + plo(q23)));
        l1 = l1 * al1 + ((phi(p01) + phi(p23)) + (phi(q01) + phi(q23)));
        m0 = mn0;
        m1 = mn1;
        bool rescale = __any_sync(0xffffffffu, grow);
        if constexpr (PSC) {
            if (vr != 1.f) {  // acc into the units of the new vref (l keeps its own)
                al0 *= vr;
                al1 *= vr;
                rescale = true;
            }
        }
        if (rescale) {
#pragma unroll
            for (int mt = 0; mt < NKK; ++mt) {
                acc[mt][0] *= al0;
                acc[mt][1] *= al1;
                acc[mt][2] *= al0;
                acc[mt][3] *= al1;
            }
        }
        if constexpr (PSC) {
            if (nva > 0) {
                if (ra != 1.f) pv8(s0a + C::KT, scale_f16x2(p01, ra), scale_f16x2(p23, ra), nva);
                else pv8(s0a + C::KT, p01, p23, nva);
            }
            if (nvb > 0) {
                if (rb != 1.f) pv8(s1a + C::KT, scale_f16x2(q01, rb), scale_f16x2(q23, rb), nvb);
                else pv8(s1a + C::KT, q01, q23, nvb);
            }
        } else if constexpr (F8) {
            if (nva > 0) pv8(s0a + C::KT, p01, p23, nva);
            if (nvb > 0) pv8(s1a + C::KT, q01, q23, nvb);
        } else {
            if (nva > 0) pv(s0a + C::KT, p01, p23, nva);
            if (nvb > 0) pv(s1a + C::KT, q01, q23, nvb);
        }
    };

    // Lane layout of the merge and the combine: the [D][8] output is 2*D
    // float4 slots (a dim and 4 heads each); lane handles slots lane + 32 r,
    // i.e. dims (lane >> 1) + 16 r for the heads h4 .. h4 + 3.
    constexpr int NSL = 2 * D / 32;  // slots per lane
    const int h4 = (lane & 1) * 4;

    // merge the CTA pieces of segment `seg` (run by one warp of the last CTA
    // to arrive), pieces in order with a running max per head; piece `own`
    // (or none: -1) comes from registers (log2-sum-exp ol, normalised ox)
    // instead of the workspace
    // pieces in slots (slot0 + i) * pst (i < pieces), output rows at ob
    auto combine = [&](int64_t slot0, int64_t pst, uint16_t *ob, int64_t s0, int64_t e0, int own,
                       const float (&ol)[4], const float4 (&ox)[NSL]) {
        const int w0 = int(s0 / L), np = int((e0 - 1) / L) - w0 + 1;
        (void)w0;
        float M[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float W[4] = {0.f, 0.f, 0.f, 0.f};
        float O[NSL][4];
#pragma unroll
        for (int r = 0; r < NSL; ++r)
#pragma unroll
            for (int e = 0; e < 4; ++e) O[r][e] = 0.f;
        constexpr int U = 2;  // pieces in flight per round
        for (int i0 = 0; i0 < np; i0 += U) {
            float4 lx[U], xv[U][NSL];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (i0 + u == own) {
                    lx[u] = make_float4(ol[0], ol[1], ol[2], ol[3]);
#pragma unroll
                    for (int r = 0; r < NSL; ++r) xv[u][r] = ox[r];
                    continue;
                }
                const float *ps = a.part + (slot0 + int64_t(min(i0 + u, np - 1)) * pst) * C::PART;
                lx[u] = __ldcg(reinterpret_cast<const float4 *>(ps + D * 8 + h4));
#pragma unroll
                for (int r = 0; r < NSL; ++r)
                    xv[u][r] = __ldcg(reinterpret_cast<const float4 *>(ps + ((lane >> 1) + 16 * r) * 8 + h4));
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                if (i0 + u >= np) break;
                const float l4[4] = {lx[u].x, lx[u].y, lx[u].z, lx[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (l4[e] == -INFINITY) continue;
                    if (l4[e] > M[e]) {
                        const float sc = fast_exp2(M[e] - l4[e]);  // 0 when M was -inf
                        W[e] *= sc;
#pragma unroll
                        for (int r = 0; r < NSL; ++r) O[r][e] *= sc;
                        M[e] = l4[e];
                    }
                    const float wt = fast_exp2(l4[e] - M[e]);
                    W[e] += wt;
#pragma unroll
                    for (int r = 0; r < NSL; ++r) {
                        const float x = e == 0 ? xv[u][r].x : e == 1 ? xv[u][r].y : e == 2 ? xv[u][r].z : xv[u][r].w;
                        O[r][e] += wt * x;
                    }
                }
            }
        }
        float iw[4];  // one reciprocal per head (32 divisions per lane took about 5 us)
#pragma unroll
        for (int e = 0; e < 4; ++e) iw[e] = W[e] > 0.f ? 1.f / W[e] : 0.f;
#pragma unroll
        for (int r = 0; r < NSL; ++r) {
            const int d = (lane >> 1) + 16 * r;
#pragma unroll
            for (int e = 0; e < 4; ++e)
                if (h4 + e < G) ob[(h4 + e) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(O[r][e] * iw[e]));
        }
    };

    // End of a segment for a consumer warp: it deposits its state in its
    // shared-memory slot and arrives on merge_bar, then goes straight on to
    // the next segment. The merge warp merges the NC states and writes the
    // CTA's piece (final output, or a partial followed by the cross-CTA
    // arrival and, for the last CTA, the combine), so no consumer holds its
    // ring stages while a merge runs.
    volatile int *read_done = flags + 2;  // instances whose states the merge warp has read
    auto deposit = [&](int inst) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
        // the slot is free once the merge warp has read the previous instance
        if (lane == 0 && *read_done < inst) {
            const uint64_t t0 = global_timer_ns();
            while (*read_done < inst) {
                if (global_timer_ns() - t0 > a.wait_ns) {
                    flags[0] = 1;
                    atomicOr(a.status, kStatusTimeout);
                    break;
                }
            }
        }
        __syncwarp();
        float *my = scr + c_id * C::SCR;
        const int hh = 2 * q4;
#pragma unroll
        for (int mt = 0; mt < NKK; ++mt) {
            const int d = 16 * mt + g;
            if constexpr (F8) {  // acc is in units of vref
                *reinterpret_cast<float2 *>(my + d * 8 + hh) = make_float2(acc[mt][0] * vref, acc[mt][1] * vref);
                *reinterpret_cast<float2 *>(my + (d + 8) * 8 + hh) =
                    make_float2(acc[mt][2] * vref, acc[mt][3] * vref);
            } else {
                *reinterpret_cast<float2 *>(my + d * 8 + hh) = make_float2(acc[mt][0], acc[mt][1]);
                *reinterpret_cast<float2 *>(my + (d + 8) * 8 + hh) = make_float2(acc[mt][2], acc[mt][3]);
            }
        }
        if (g == 0) {
            *reinterpret_cast<float2 *>(my + D * 8 + hh) = make_float2(m0, m1);
            *reinterpret_cast<float2 *>(my + D * 8 + 8 + hh) = make_float2(l0, l1);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(merge_bar);  // release: the slot's writes precede the arrival
    };

    // the merge warp's part of segment seg's end: the NC deposited states
    // (instance inst) merged into the CTA's piece
    auto merge_states = [&](int seg, int64_t s0, int64_t e0, bool whole, int inst) {
        if (!mbar_wait_bounded(merge_bar, uint32_t(inst & 1), a.wait_ns)) {
            if (lane == 0) {
                flags[0] = 1;
                atomicOr(a.status, kStatusTimeout);
            }
            return false;
        }
        // pieces of a split segment already counted (read while merging)
        int seen = 0;
        if (!whole && lane == 0) seen = ld_acquire_s32(a.counters + seg);
        float M[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
        float mc[NC][4], lc[NC][4];
#pragma unroll
        for (int cc = 0; cc < NC; ++cc) {
            const float4 mm = *reinterpret_cast<const float4 *>(scr + cc * C::SCR + D * 8 + h4);
            const float4 ll = *reinterpret_cast<const float4 *>(scr + cc * C::SCR + D * 8 + 8 + h4);
            mc[cc][0] = mm.x; mc[cc][1] = mm.y; mc[cc][2] = mm.z; mc[cc][3] = mm.w;
            lc[cc][0] = ll.x; lc[cc][1] = ll.y; lc[cc][2] = ll.z; lc[cc][3] = ll.w;
#pragma unroll
            for (int e = 0; e < 4; ++e) M[e] = fmaxf(M[e], mc[cc][e]);
        }
        float Ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cc = 0; cc < NC; ++cc)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                mc[cc][e] = (mc[cc][e] == -INFINITY) ? 0.f : fast_exp2(mc[cc][e] - M[e]);  // weight
                Ls[e] += mc[cc][e] * lc[cc][e];
            }
        float O[NSL][4];
#pragma unroll
        for (int r = 0; r < NSL; ++r) {
            const int d = (lane >> 1) + 16 * r;
#pragma unroll
            for (int e = 0; e < 4; ++e) O[r][e] = 0.f;
#pragma unroll
            for (int cc = 0; cc < NC; ++cc) {
                const float4 xx = *reinterpret_cast<const float4 *>(scr + cc * C::SCR + d * 8 + h4);
                O[r][0] += mc[cc][0] * xx.x;
                O[r][1] += mc[cc][1] * xx.y;
                O[r][2] += mc[cc][2] * xx.z;
                O[r][3] += mc[cc][3] * xx.w;
            }
        }
        __syncwarp();
        if (lane == 0) {
            __threadfence_block();
            *read_done = inst + 1;  // the slots may be written again
        }
        const int b = seg / Hkv, kvh = seg % Hkv;
        // one reciprocal per head, then products: 32 divisions per lane here
        // held a merge for about 5 us
        float inv[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) inv[e] = Ls[e] > 0.f ? 1.f / Ls[e] : 0.f;
        if (whole) {
            uint16_t *ob = a.out + (int64_t(b) * a.Hq + kvh * G) * D;
#pragma unroll
            for (int r = 0; r < NSL; ++r) {
                const int d = (lane >> 1) + 16 * r;
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (h4 + e < G) ob[(h4 + e) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(O[r][e] * inv[e]));
            }
            return true;
        }
        // this CTA's piece, normalised, and its log2-sum-exp
        float lse[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) lse[e] = Ls[e] > 0.f ? M[e] + log2f(Ls[e]) : -INFINITY;
        float4 ox[NSL];
#pragma unroll
        for (int r = 0; r < NSL; ++r)
            ox[r] = make_float4(O[r][0] * inv[0], O[r][1] * inv[1], O[r][2] * inv[2], O[r][3] * inv[3]);
        const int w0 = int(s0 / L);
        const int npieces = int((e0 - 1) / L) - w0 + 1;
        seen = __shfl_sync(0xffffffffu, seen, 0);
        if (seen == npieces - 1) {
            // Every other piece has been counted, so this one completes the
            // segment: combine from registers, without publishing it. Lane 0
            // read the count with acquire semantics, and the warp barrier
            // orders every lane's loads of the counted pieces after it (a
            // full GPU fence here held the merge warp for 5-9 us).
            __syncwarp();
            combine(int64_t(seg) + w0, 1, a.out + (int64_t(seg / Hkv) * a.Hq + (seg % Hkv) * G) * D, s0, e0,
                    int(blockIdx.x) - w0, lse, ox);
            if (lane == 0) a.counters[seg] = 0;
            return true;
        }
        float *ps = a.part + int64_t(seg + blockIdx.x) * C::PART;
#pragma unroll
        for (int r = 0; r < NSL; ++r) {
            const int d = (lane >> 1) + 16 * r;
            __stcg(reinterpret_cast<float4 *>(ps + d * 8 + h4), ox[r]);
        }
        if (lane < 2)
            __stcg(reinterpret_cast<float4 *>(ps + D * 8 + h4), make_float4(lse[0], lse[1], lse[2], lse[3]));
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            // release this CTA's partial (written by the warp, ordered by the
            // warp barrier) and acquire the pieces counted before it
            __threadfence_block();
            last = (atomic_add_acq_rel_gpu(a.counters + seg, 1) == npieces - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();  // every lane's reads of the pieces follow lane 0's acquire
        if (last) {
            const float nol[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            combine(int64_t(seg) + w0, 1, a.out + (int64_t(seg / Hkv) * a.Hq + (seg % Hkv) * G) * D, s0, e0,
                    -1, nol, ox);
            if (lane == 0) a.counters[seg] = 0;
        }
        return true;
    };

    // MULTI: end of a piece [s0, e0) of work-list segment seg for this
    // consumer's own query row `row` (slot index (segment + CTA) * RG + c_id;
    // counter segment * RG + c_id): the whole segment writes the row's bf16
    // output from the registers, otherwise a normalised partial and its lse,
    // and the piece that completes the count combines.
    auto finish_row = [&](int seg, int row, int64_t s0, int64_t e0, bool whole) {
        l0 += __shfl_xor_sync(0xffffffffu, l0, 4);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 8);
        l0 += __shfl_xor_sync(0xffffffffu, l0, 16);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 4);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 8);
        l1 += __shfl_xor_sync(0xffffffffu, l1, 16);
        const int kvh = seg % Hkv, h0 = 2 * q4;
        const float inv0 = l0 > 0.f ? 1.f / l0 : 0.f, inv1 = l1 > 0.f ? 1.f / l1 : 0.f;
        uint16_t *ob = a.out + (int64_t(row) * a.Hq + kvh * G) * D;
        if (whole) {
#pragma unroll
            for (int mt = 0; mt < NKK; ++mt) {
                const int d = 16 * mt + g;
                if (h0 < G) {
                    ob[h0 * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][0] * inv0));
                    ob[h0 * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][2] * inv0));
                }
                if (h0 + 1 < G) {
                    ob[(h0 + 1) * D + d] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][1] * inv1));
                    ob[(h0 + 1) * D + d + 8] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[mt][3] * inv1));
                }
            }
            return;
        }
        const int w0 = int(s0 / L);
        const int npieces = int((e0 - 1) / L) - w0 + 1;
        float *ps = a.part + ((int64_t(seg) + blockIdx.x) * RG + c_id) * C::PART;
#pragma unroll
        for (int mt = 0; mt < NKK; ++mt) {
            const int d = 16 * mt + g;
            __stcg(reinterpret_cast<float2 *>(ps + d * 8 + h0), make_float2(acc[mt][0] * inv0, acc[mt][1] * inv1));
            __stcg(reinterpret_cast<float2 *>(ps + (d + 8) * 8 + h0),
                   make_float2(acc[mt][2] * inv0, acc[mt][3] * inv1));
        }
        if (g == 0)
            __stcg(reinterpret_cast<float2 *>(ps + D * 8 + h0),
                   make_float2(l0 > 0.f ? m0 + log2f(l0) : -INFINITY, l1 > 0.f ? m1 + log2f(l1) : -INFINITY));
        __syncwarp();
        int last = 0;
        if (lane == 0) {
            __threadfence_block();
            last = (atomic_add_acq_rel_gpu(a.counters + int64_t(seg) * RG + c_id, 1) == npieces - 1);
        }
        last = __shfl_sync(0xffffffffu, last, 0);
        __syncwarp();
        if (last) {
            const float nol[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
            float4 dummy[NSL];
#pragma unroll
            for (int r = 0; r < NSL; ++r) dummy[r] = make_float4(0.f, 0.f, 0.f, 0.f);
            combine((int64_t(seg) + w0) * RG + c_id, RG, ob, s0, e0, -1, nol, dummy);
            if (lane == 0) a.counters[int64_t(seg) * RG + c_id] = 0;
        }
    };

    if constexpr (MULTI) {
        // every consumer streams every item of the segment for its own query row
        int64_t p = pos0;
        int b = find_seq(p);
        int kvh = int((p - int64_t(Hkv) * pre[b]) / (pre[b + 1] - pre[b]));
        while (p < pos1) {
            const int n = pre[b + 1] - pre[b];
            const int seg = b * Hkv + kvh;
            const int64_t s0 = int64_t(Hkv) * pre[b] + int64_t(kvh) * n;
            const int64_t e0 = s0 + n;
            const int ks0 = int(p - pos0), ks1 = int(min(e0, pos1) - pos0);
            const int sq = seq_of[b], row = row0_of[b] + c_id;
            const bool act = row < __ldg(a.cu_q + sq + 1) && row < B;
            const int lim = act ? row_ctx(row, sq) : 0;
            load_q(seg, act ? row : -1);
            for (int ka = ks0; ka < ks1; ka += 2) {
                const int kb = min(ka + 1, ks1 - 1);
                int ja = 0, jb = 0;
                int nva = wait_full_j(ka, ja);
                int nvb = (kb > ka) ? wait_full_j(kb, jb) : 0;
                nva = act ? min(nva, max(lim - ja * BS, 0)) : 0;
                nvb = act ? min(nvb, max(lim - jb * BS, 0)) : 0;
                if (nva > 0 || nvb > 0)
                    step(base + (ka % S) * C::STAGE, nva, float2{}, base + (kb % S) * C::STAGE, nvb, float2{});
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar + (ka % S) * 8);
                    if (kb > ka) mbar_arrive(empty_bar + (kb % S) * 8);
                }
            }
            if (act) finish_row(seg, row, s0, e0, (s0 >= pos0) && (e0 <= pos1));
            p = min(e0, pos1);
            if (++kvh == Hkv) {
                kvh = 0;
                do {
                    ++b;
                } while (b < NR && pre[b + 1] == pre[b]);
            }
        }
        return;
    }

    // walk the segments of this CTA's range in order: the consumers stream
    // each segment's items and deposit their states, the merge warp merges
    // them (instance inst = segments finished so far, the same count in
    // every warp)
    const bool merge_warp = warp == NC + 1;
    if (merge_warp && early) pdl_wait();  // before its first write
    int64_t p = pos0;
    int inst = 0;
    int b = find_seq(p);
    int kvh = int((p - int64_t(Hkv) * pre[b]) / (pre[b + 1] - pre[b]));
    while (p < pos1) {
        const int n = pre[b + 1] - pre[b];
        const int seg = b * Hkv + kvh;
        const int64_t s0 = int64_t(Hkv) * pre[b] + int64_t(kvh) * n;
        const int64_t e0 = s0 + n;
        const int ks0 = int(p - pos0), ks1 = int(min(e0, pos1) - pos0);
        const bool whole = (s0 >= pos0) && (e0 <= pos1);
        if (merge_warp) {
            if (!merge_states(seg, s0, e0, whole, inst++)) return;
            p = min(e0, pos1);
            if (++kvh == Hkv) {
                kvh = 0;
                do {
                    ++b;
                } while (b < NR && pre[b + 1] == pre[b]);
            }
            continue;
        }
        load_q(seg, b);
        if constexpr (F8) {
            // two-block items of this segment owned by this warp: k % NC == c_id
            for (int k = ks0 + (c_id - ks0 % NC + NC) % NC; k < ks1; k += NC) {
                const int nvp = wait_full(k);
                const int nva = nvp & 255, nvb = nvp >> 8;
                const uint32_t sa = base + (k % S) * C::STAGE;
                float4 sc4 = make_float4(0.f, 0.f, 0.f, 0.f);
                if constexpr (PSC) sc4 = iscale[k % S];
                if (nva > 0 || nvb > 0)
                    step(sa, nva, make_float2(sc4.x, sc4.y), sa + 2 * C::KT, nvb, make_float2(sc4.z, sc4.w));
                __syncwarp();
                if (lane == 0) mbar_arrive(empty_bar + (k % S) * 8);
            }
        } else {
            // item pairs (2q, 2q+1) of this segment owned by this warp: q % NC == c_id
            int q = ks0 >> 1;
            q += (c_id - q % NC + NC) % NC;
            for (; 2 * q < ks1; q += NC) {
                const int ka = max(2 * q, ks0);
                const int kb = min(2 * q + 1, ks1 - 1);
                const int nva = wait_full(ka);
                const int nvb = (kb > ka) ? wait_full(kb) : 0;
                if (nva > 0 || nvb > 0)
                    step(base + (ka % S) * C::STAGE, nva, float2{}, base + (kb % S) * C::STAGE, nvb, float2{});
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(empty_bar + (ka % S) * 8);
                    if (kb > ka) mbar_arrive(empty_bar + (kb % S) * 8);
                }
            }
        }
        deposit(inst++);
        p = min(e0, pos1);
        if (++kvh == Hkv) {
            kvh = 0;
            do {
                ++b;
            } while (b < NR && pre[b + 1] == pre[b]);
        }
    }
}

template <int D, bool F8>
cudaError_t geometry_t(DecodeGeometry *g) {
    using C = DecodeCfg<D, F8>;
    using CM = DecodeCfg<D, F8, true>;
    cudaError_t e;
    int dev = 0, sms = 0, per_sm = 0, optin = 0;
    if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
        return e;
    // shared memory for the largest batch that fits (the ring is fixed; the
    // per-sequence prefix grows with the batch)
    const size_t smem = C::smem_bytes(kMaxBatch) < size_t(optin) ? C::smem_bytes(kMaxBatch) : size_t(optin);
    const size_t smem_m = CM::smem_bytes(kMaxBatch) < size_t(optin) ? CM::smem_bytes(kMaxBatch) : size_t(optin);
    if (smem < C::smem_bytes(1)) return cudaErrorInvalidConfiguration;
    // the second kernel: multi-token rows (bf16), or per-block scales (E4M3)
    void (*kernels[2])(CUtensorMap, CUtensorMap, DecodeArgs) = {decode_kernel<D, F8, false>,
                                                                decode_kernel<D, F8, !F8, F8>};
    const size_t limits[2] = {smem, F8 ? smem : smem_m};
    for (int i = 0; i < 2; ++i) {
        e = cudaFuncSetAttribute(kernels[i], cudaFuncAttributeMaxDynamicSharedMemorySize, int(limits[i]));
        if (e != cudaSuccess) return e;
        // same L1/shared split as the library's other kernels: no reconfiguration between them
        cudaFuncSetAttribute(kernels[i], cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    }
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<D, F8, false>, C::THREADS,
                                                      smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    g->grid = sms * per_sm;
    g->warps = C::NC + 1;
    g->workers = g->grid;
    g->smem = smem;
    g->smem_multi = smem_m;
    return cudaSuccess;
}

template <int D, bool SPARSE, bool F8, bool MULTI = false, bool BSC = false>
cudaError_t launch_t(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                     cudaStream_t stream, int max_ctas = 0) {
    using C = DecodeCfg<D, F8, MULTI>;
    DecodeGeometry geo;
    cudaError_t e = decode_geometry(D, &geo, F8);
    if (e != cudaSuccess) return e;
    const size_t smem = MULTI ? C::smem_bytes(a.B > a.nseq ? a.B : a.nseq, a.B) : C::smem_bytes(a.B);
    if (smem > (MULTI ? geo.smem_multi : geo.smem)) return cudaErrorInvalidConfiguration;  // batch too large
    int grid = geo.grid;
    if (SPARSE) {
        // Every non-empty (sequence, KV head) segment has exactly topk items,
        // known here. For small selections a CTA holding a few items spends
        // most of its time on fixed costs (start-up, publishing partials, the
        // cross-CTA combine), and a range boundary inside a segment costs a
        // combine: cut each segment into c equal pieces (c a power of two, at
        // least kSparseMinItems items each, at most `budget` CTAs in all) or
        // give each CTA whole segments. The budget is the caller's max_ctas;
        // by default half the SMs when the segments fit in it, else one CTA
        // per SM. A piece boundary costs a partial and a combine, and in the
        // fused Quest decode every piece repeats its segment's top-K: on
        // quest_8k (64 segments of 64 blocks) 64 CTAs took 41.0 us against
        // 45.1 us for 128 (quest_decode), with the sparse decode alone equal;
        // dense_b32's 128 segments need 128 CTAs (43.0 against 57.3 us).
        // In a step that runs the sparse decode beside the dense one, half
        // the SMs also let it start on the SMs the dense CTAs free without
        // waiting for the last of them (quest_8k step 83.6 -> 77.3 us).
        const int64_t segs = int64_t(a.B) * a.Hkv;
        const int budget = (max_ctas > 0 && max_ctas < grid) ? max_ctas : (segs <= grid / 2 ? grid / 2 : grid);
        const int tk = (a.topk + C::BPI - 1) / C::BPI;  // items per segment
        if (segs * a.topk < int64_t(grid) * kSparseLargeItems) {
            int64_t c = 1;
            while (tk % (2 * c) == 0 && a.topk / (2 * c) >= kSparseMinItems && segs * 2 * c <= budget)
                c *= 2;
            if (segs * c <= budget) {
                grid = int(segs * c);
            } else {
                const int64_t m = (segs + budget - 1) / budget;  // segments per CTA
                grid = int((segs + m - 1) / m);
            }
        } else {
            grid = budget;
        }
    } else if (max_ctas > 0 && max_ctas < grid) {
        // dense: the caller's CTA budget, so that other work can run on the
        // remaining SMs (the work list is cut into max_ctas equal ranges)
        grid = max_ctas;
    }
    if (SPARSE && a.scores) {
        // fused Quest decode: room for the CTA's selection entries (at most
        // BPI * ceil(items / CTAs), items <= segments * ceil(topk / BPI))
        DecodeArgs f = a;
        const int64_t items = int64_t(a.B) * a.Hkv * ((a.topk + C::BPI - 1) / C::BPI);
        const int64_t cap = C::BPI * ((items + grid - 1) / grid);
        const size_t fsmem = C::smem_bytes_sel(a.B, int(cap));
        if (cap > (int64_t(1) << 20) || fsmem > geo.smem) return cudaErrorInvalidConfiguration;
        f.nsel_cap = int(cap);
        return launch_pdl(decode_kernel<D, F8, MULTI, BSC>, dim3(grid), dim3(C::THREADS), fsmem, stream, tm_k, tm_v,
                          f);
    }
    return launch_pdl(decode_kernel<D, F8, MULTI, BSC>, dim3(grid), dim3(C::THREADS), smem, stream,
                      tm_k, tm_v, a);
}

constexpr int kMaxDevices = 64;
DecodeGeometry g_geo[kMaxDevices][3];  // head_dim 64, 128, 128 with an E4M3 cache
bool g_geo_ok[kMaxDevices][3];

}  // namespace

cudaError_t decode_geometry(int head_dim, DecodeGeometry *g, bool fp8) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    if (fp8 && head_dim != 128) return cudaErrorInvalidValue;
    const int idx = fp8 ? 2 : (head_dim == 128 ? 1 : 0);
    if (!g_geo_ok[dev][idx]) {
        DecodeGeometry t{};
        e = fp8 ? geometry_t<128, true>(&t)
                : (head_dim == 128 ? geometry_t<128, false>(&t) : geometry_t<64, false>(&t));
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

// multi-token rows: one counter and one partial slot per (segment, query row of its group)
size_t decode_multi_workspace_bytes(int total_q, int Hkv, int head_dim, int workers) {
    const int RG = kMultiRowGroup;
    const size_t segs = size_t(total_q) * Hkv;
    const size_t counters = (segs * RG * 4 + 255) / 256 * 256;
    return 256 + counters + (segs + size_t(workers)) * RG * size_t(head_dim * 8 + 8) * 4;
}

cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                          int head_dim, bool sparse, cudaStream_t stream, bool fp8, int max_ctas) {
    if (a.cu_q) {  // multi-token query rows (bf16 cache, dense)
        if (fp8 || sparse) return cudaErrorInvalidValue;
        return head_dim == 128 ? launch_t<128, false, false, true>(tm_k, tm_v, a, stream, max_ctas)
                               : launch_t<64, false, false, true>(tm_k, tm_v, a, stream, max_ctas);
    }
    if (fp8) {
        if (head_dim != 128) return cudaErrorInvalidValue;
        if (a.scale_per_block)
            return sparse ? launch_t<128, true, true, false, true>(tm_k, tm_v, a, stream, max_ctas)
                          : launch_t<128, false, true, false, true>(tm_k, tm_v, a, stream, max_ctas);
        return sparse ? launch_t<128, true, true>(tm_k, tm_v, a, stream, max_ctas)
                      : launch_t<128, false, true>(tm_k, tm_v, a, stream, max_ctas);
    }
    if (head_dim == 128)
        return sparse ? launch_t<128, true, false>(tm_k, tm_v, a, stream, max_ctas)
                      : launch_t<128, false, false>(tm_k, tm_v, a, stream, max_ctas);
    return sparse ? launch_t<64, true, false>(tm_k, tm_v, a, stream, max_ctas)
                  : launch_t<64, false, false>(tm_k, tm_v, a, stream, max_ctas);
}

}  // namespace pa
