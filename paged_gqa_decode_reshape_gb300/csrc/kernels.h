// kernels.h -- internal interface between the C-ABI layer and the kernels.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kBlockSize = 16;       // tokens per KV block
constexpr int kMaxBatch = 4096;      // sequences per call
constexpr int kMaxGroup = 8;         // query heads per KV head (one mma n-tile)
constexpr int kMaxMultiRows = 2048;  // query rows of a multi-token decode call
constexpr int kMultiRowGroup = 4;    // query rows sharing one pass over the KV (one per consumer warp)
// Sparse decode of small selections (fewer than kSparseLargeItems items per
// SM): the grid follows the segments instead of cutting one work list evenly
constexpr int kSparseLargeItems = 96;

// Arguments of the split-KV decode kernel (dense and Quest-sparse).
struct DecodeArgs {
    const uint16_t *q;          // [B][Hq][D] bf16
    const int32_t *bt;          // [B][MBS]
    const int32_t *ctx;         // [B]
    const int32_t *sel;         // [B][Hkv][topk] (sparse only)
    const float *k_scale;       // scales of an E4M3 cache (else null): [Hkv] per KV head,
    const float *v_scale;       // or [NB][Hkv] per physical block when scale_per_block
    int scale_per_block;
    const uint8_t *v8;          // E4M3 V cache [NB][Hkv][D][16] (else null): tiles are contiguous
    const int32_t *cu_q;        // multi-token rows: [nseq + 1] row offsets per sequence (else null;
                                // B then counts query rows, ctx / bt are per sequence)
    int nseq;
    uint16_t *out;              // [B][Hq][D] bf16
    float *part;                // [B*Hkv + W][D*8 + 8] partial outputs and lse (log2 domain)
    int32_t *counters;          // [B*Hkv] arrival counters (zero between calls)
    int32_t *status;            // workspace status word
    const float *scores;        // fused Quest decode: block scores [B][Hkv][MBS]; each CTA selects
                                // the top-K of its segments itself (else null: selection in sel)
    int32_t *sel_out;           // fused Quest decode: [B][Hkv][topk] selection written out
    int nsel_cap;               // fused Quest decode: capacity of the CTA's selection array
    // dense decode with the step's write (bf16 cache, one query row): token b's
    // K and V rows ([B][Hkv][D]) go to slot new_slots[b] when that is the
    // slot of position ctx_b - 1 of sequence b; the CTA that reads the block
    // writes its KV head's slice first (and the metadata when kmin_w is set)
    const uint16_t *new_k, *new_v;
    const int64_t *new_slots;
    uint16_t *kc_w, *vc_w, *kmin_w, *kmax_w;
    uint64_t wait_ns;           // limit of every bounded wait inside the kernel (ns)
    int stop_item;              // the producer stops issuing at this item of its CTA's range
                                // (failure tests only; INT_MAX otherwise)
    int64_t NB;
    int MBS, topk, B, Hq, Hkv, G;
    float scale_log2;           // softmax scale * log2(e)
};

// Per-device launch geometry of the decode kernel for one head_dim.
struct DecodeGeometry {
    int grid;          // CTAs (persistent)
    int warps;         // warps per CTA
    int workers;       // grid * warps
    size_t smem;       // dynamic shared memory limit set on the kernel (one query row per sequence)
    size_t smem_multi; // the same for the multi-token kernel
};

cudaError_t decode_geometry(int head_dim, DecodeGeometry *g, bool fp8 = false);
size_t decode_workspace_bytes(int B, int Hkv, int head_dim, int workers);
size_t decode_multi_workspace_bytes(int total_q, int Hkv, int head_dim, int workers);
// max_ctas: at most this many CTAs. Sparse: <= 0 gives half the SMs when the
// segments fit in them, else one per SM. Dense: <= 0 gives one per SM.
cudaError_t launch_decode(const CUtensorMap &tm_k, const CUtensorMap &tm_v, const DecodeArgs &a,
                          int head_dim, bool sparse, cudaStream_t stream, bool fp8 = false,
                          int max_ctas = 0);

cudaError_t launch_reshape_and_cache(const uint16_t *key, const uint16_t *value, uint16_t *kc,
                                     uint16_t *vc, const int64_t *slots, int64_t T, int Hkv, int D,
                                     int BS, int64_t NB, cudaStream_t stream);
cudaError_t launch_update_meta(uint16_t *kmin, uint16_t *kmax, const uint16_t *key,
                               const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                               cudaStream_t stream);
cudaError_t launch_write_quest(uint16_t *kc, uint16_t *vc, uint16_t *kmin, uint16_t *kmax,
                               const uint16_t *key, const uint16_t *value, const int64_t *slots,
                               int64_t T, int Hkv, int D, int BS, int64_t NB, cudaStream_t stream);
cudaError_t launch_rebuild_meta(uint16_t *kmin, uint16_t *kmax, const uint16_t *kc,
                                const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hkv,
                                int D, int BS, int64_t NB, cudaStream_t stream);
cudaError_t launch_check_metadata(int32_t *counts, const int64_t *slots, int64_t T,
                                  const int32_t *bt, int MBS, const int32_t *ctx, int B, int BS,
                                  int64_t NB, cudaStream_t stream);

cudaError_t launch_write_fp8(uint8_t *kc, uint8_t *vc, uint8_t *kmin, uint8_t *kmax, const uint16_t *key,
                             const uint16_t *value, const float *k_scale, const float *v_scale,
                             const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                             cudaStream_t stream);
cudaError_t launch_update_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint16_t *key, const float *k_scale,
                                   const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                                   cudaStream_t stream);
cudaError_t launch_rebuild_meta_fp8(uint8_t *kmin, uint8_t *kmax, const uint8_t *kc, const int32_t *bt,
                                    int MBS, const int32_t *ctx, int B, int Hkv, int D, int BS, int64_t NB,
                                    cudaStream_t stream);

// E4M3 cache with per-block scales: ReshapeAndCache (and the metadata when
// kmin is not null) with the scales k_bscale / v_bscale [NB][Hkv] kept up to
// date (powers of two; 0 for an empty block)
cudaError_t launch_write_fp8_block(uint8_t *kc, uint8_t *vc, uint8_t *kmin, uint8_t *kmax, float *k_bscale,
                                   float *v_bscale, const uint16_t *key, const uint16_t *value,
                                   const int64_t *slots, int64_t T, int Hkv, int D, int BS, int64_t NB,
                                   cudaStream_t stream);

// The step's write folded into the score launch (bf16 cache): the warp that
// scores the chunk holding sequence b's block of position ctx_b - 1 writes
// token b's KV-head slice there (when slots[b] is that slot) and updates the
// block's metadata before scoring it.
struct ScoreWrite {
    const uint16_t *key, *value;  // [B][Hkv][D] bf16
    const int64_t *slots;         // [B]
    uint16_t *kc, *vc;            // the caches
    uint16_t *kmin, *kmax;        // the metadata (the score kernel's kmin / kmax)
};

// block scores only (the first launch of the fused Quest decode)
// k_bscale: per-block K scales [NB][Hkv] of an E4M3 cache (else null)
cudaError_t launch_quest_scores(float *scores, const uint16_t *q, const void *kmin, const void *kmax,
                                const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hq, int Hkv, int D,
                                int BS, int64_t NB, cudaStream_t stream, bool fp8 = false,
                                const float *k_bscale = nullptr, const ScoreWrite *write = nullptr);
// kmin / kmax: bf16 metadata, or E4M3 codes when fp8 (head_dim 128)
cudaError_t launch_quest_select(int32_t *sel, float *scores, const uint16_t *q, const void *kmin,
                                const void *kmax, const int32_t *bt, int MBS, const int32_t *ctx,
                                int B, int Hq, int Hkv, int D, int BS, int64_t NB, int topk,
                                cudaStream_t stream, bool fp8 = false, const float *k_bscale = nullptr,
                                const ScoreWrite *write = nullptr);

}  // namespace pa
