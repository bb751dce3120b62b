// api.cu -- the C ABI (include/paged_decode.h): argument checks on the host,
// TMA descriptors, workspace carving, and the kernel launches. Nothing here
// allocates device memory.
#include <atomic>
#include <climits>
#include <cstring>

#include "../../include/paged_decode.h"
#include "kernels.h"

using namespace pa;

namespace {

thread_local int g_last_cuda_error = 0;

// Limit of every bounded wait inside the decode kernel, and the item at which
// its producer stops issuing copies. Fixed at 0.5 s and "never" in the
// library; the failure-test build (PA_FAULT_TEST) lets a test change both, so
// that a wait runs out on purpose and the timeout path can be checked.
constexpr uint64_t kDefaultWaitNs = 500ull * 1000ull * 1000ull;
std::atomic<uint64_t> g_wait_ns{kDefaultWaitNs};
std::atomic<int> g_stop_item{INT_MAX};

int cuda_fail(cudaError_t e) {
    g_last_cuda_error = int(e);
    return PA_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

bool shape_supported(int head_dim, int block_size) {
    return (head_dim == 64 || head_dim == 128) && block_size == kBlockSize;
}

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link
// against libcuda needed).
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static const EncodeTiledFn fn = [] {  // looked up once (thread-safe initialisation)
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            return reinterpret_cast<EncodeTiledFn>(p);
        return EncodeTiledFn(nullptr);
    }();
    return fn;
}

// Tensor map over one layer's paged cache [NB][BS][Hkv][D], boxes of
// [1 block][BS tokens][1 head][128 bytes of dims] with 128-byte swizzle:
// 64 bf16 dims, or 128 E4M3 codes (fp8).
int make_cache_map(CUtensorMap *map, const void *cache, int Hkv, int D, int BS, int64_t NB,
                   bool fp8 = false) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail(cudaErrorNotSupported);
    const cuuint64_t eb = fp8 ? 1 : 2;
    const cuuint64_t dims[4] = {cuuint64_t(D), cuuint64_t(Hkv), cuuint64_t(BS), cuuint64_t(NB)};
    const cuuint64_t strides[3] = {cuuint64_t(D) * eb, cuuint64_t(Hkv) * D * eb,
                                   cuuint64_t(BS) * Hkv * D * eb};
    const cuuint32_t box[4] = {fp8 ? 128u : 64u, 1u, cuuint32_t(BS), 1u};
    const cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    // bf16: the two 128-byte halves of a row belong to the same tile, so L2
    // fills of 256 bytes waste nothing; an E4M3 row is 128 bytes and its
    // neighbour belongs to another KV head, so fills stay at 128 bytes.
    const CUresult r = fn(map, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                          const_cast<void *>(cache), dims,
                          strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B,
                          fp8 ? CU_TENSOR_MAP_L2_PROMOTION_L2_128B : CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cuda_fail(cudaErrorInvalidValue);
    return PA_OK;
}

struct DecodeWorkspace {
    int32_t *status;
    int32_t *counters;
    float *part;
};

DecodeWorkspace carve_decode_ws(void *ws, int B, int Hkv, int per_seg = 1) {
    uint8_t *p = static_cast<uint8_t *>(ws);
    const size_t segs = size_t(B) * Hkv;
    const size_t counters = (segs * per_seg * 4 + 255) / 256 * 256;
    DecodeWorkspace d;
    d.status = reinterpret_cast<int32_t *>(p);
    d.counters = reinterpret_cast<int32_t *>(p + 256);
    d.part = reinterpret_cast<float *>(p + 256 + counters);
    return d;
}

int check_attention_args(const void *out, const void *q, const void *kc, const void *vc,
                         const int32_t *bt, int MBS, const int32_t *ctx, int B, int Hq, int Hkv,
                         int D, int BS, int64_t NB, float scale, const void *ws) {
    if (!out || !q || !kc || !vc || !bt || !ctx || !ws) return PA_ERR_INVALID_ARG;
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || BS <= 0 || NB <= 0 || MBS <= 0)
        return PA_ERR_INVALID_ARG;
    if (Hq % Hkv != 0) return PA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return PA_ERR_INVALID_ARG;
    if (!shape_supported(D, BS) || Hq / Hkv > kMaxGroup || B > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if (int64_t(MBS) * BS > int64_t(1) << 30) return PA_ERR_UNSUPPORTED;
    if (NB > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    if (!aligned16(out) || !aligned16(q) || !aligned16(kc) || !aligned16(vc) || !aligned16(ws))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

int run_decode(pa_bf16 *out, const pa_bf16 *query, const void *key_cache, const void *value_cache,
               const int32_t *block_tables, int MBS, const int32_t *context_lens,
               const int32_t *selected, int topk, int B, int Hq, int Hkv, int D, int BS, int64_t NB,
               float scale, void *workspace, size_t workspace_bytes, void *stream, bool sparse,
               const float *k_scale = nullptr, const float *v_scale = nullptr, bool fp8 = false,
               const int32_t *cu_q = nullptr, int nseq = 0, int max_ctas = 0,
               const float *scores = nullptr, int32_t *sel_out = nullptr, bool bscale = false,
               const ScoreWrite *sw = nullptr) {
    int rc = check_attention_args(out, query, key_cache, value_cache, block_tables, MBS,
                                  context_lens, B, Hq, Hkv, D, BS, NB, scale, workspace);
    if (rc != PA_OK) return rc;
    if (sparse && ((!selected && !scores) || topk <= 0)) return PA_ERR_INVALID_ARG;
    if (fp8 && (!k_scale || !v_scale)) return PA_ERR_INVALID_ARG;
    if (fp8 && D != 128) return PA_ERR_UNSUPPORTED;
    DecodeGeometry geo;
    cudaError_t e = decode_geometry(D, &geo, fp8);
    if (e != cudaSuccess) return cuda_fail(e);
    const size_t need = cu_q ? decode_multi_workspace_bytes(B, Hkv, D, geo.workers)
                             : decode_workspace_bytes(B, Hkv, D, geo.workers);
    if (workspace_bytes < need) return PA_ERR_WORKSPACE;
    CUtensorMap tk, tv;
    if ((rc = make_cache_map(&tk, key_cache, Hkv, D, BS, NB, fp8)) != PA_OK) return rc;
    // an E4M3 V cache is read with plain bulk copies (its tiles are contiguous)
    if (fp8) std::memset(&tv, 0, sizeof tv);
    else if ((rc = make_cache_map(&tv, value_cache, Hkv, D, BS, NB)) != PA_OK) return rc;
    const DecodeWorkspace w = carve_decode_ws(workspace, B, Hkv, cu_q ? kMultiRowGroup : 1);
    DecodeArgs a;
    a.q = query;
    a.bt = block_tables;
    a.ctx = context_lens;
    a.sel = selected;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.scale_per_block = bscale ? 1 : 0;
    a.v8 = fp8 ? static_cast<const uint8_t *>(value_cache) : nullptr;
    a.cu_q = cu_q;
    a.nseq = cu_q ? nseq : B;
    a.out = out;
    a.part = w.part;
    a.counters = w.counters;
    a.status = w.status;
    a.scores = scores;
    a.sel_out = sel_out;
    a.new_k = sw ? sw->key : nullptr;  // dense decode with the step's write
    a.new_v = sw ? sw->value : nullptr;
    a.new_slots = sw ? sw->slots : nullptr;
    a.kc_w = sw ? sw->kc : nullptr;
    a.vc_w = sw ? sw->vc : nullptr;
    a.kmin_w = sw ? sw->kmin : nullptr;
    a.kmax_w = sw ? sw->kmax : nullptr;
    a.nsel_cap = 0;
    a.wait_ns = g_wait_ns.load(std::memory_order_relaxed);
    a.stop_item = g_stop_item.load(std::memory_order_relaxed);
    a.NB = NB;
    a.MBS = MBS;
    a.topk = sparse ? topk : 0;
    a.B = B;
    a.Hq = Hq;
    a.Hkv = Hkv;
    a.G = Hq / Hkv;
    a.scale_log2 = scale * 1.4426950408889634f;
    e = launch_decode(tk, tv, a, D, sparse, static_cast<cudaStream_t>(stream), fp8, max_ctas);
    if (e != cudaSuccess) return cuda_fail(e);
    return PA_OK;
}

}  // namespace

extern "C" {

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "PA_OK";
        case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG";
        case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
        case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
        case PA_ERR_CUDA: return "PA_ERR_CUDA";
        case PA_ERR_DEVICE: return "PA_ERR_DEVICE";
        default: return "PA_ERR_UNKNOWN";
    }
}

int pa_last_cuda_error(void) { return g_last_cuda_error; }

int pa_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *key_cache,
                         pa_bf16 *value_cache, const int64_t *slot_mapping, int64_t num_tokens,
                         int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                         void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!shape_supported(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_reshape_and_cache(key, value, key_cache, value_cache, slot_mapping,
                                                   num_tokens, num_kv_heads, head_dim, block_size,
                                                   num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t pa_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim) {
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0)
        return 0;
    if (!shape_supported(head_dim, kBlockSize) || batch > kMaxBatch) return 0;
    DecodeGeometry geo;
    if (decode_geometry(head_dim, &geo) != cudaSuccess) return 0;
    return decode_workspace_bytes(batch, num_kv_heads, head_dim, geo.workers);
}

int pa_decode(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
              const pa_bf16 *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
              const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
              int head_dim, int block_size, int64_t num_blocks, float scale, void *workspace,
              size_t workspace_bytes, void *stream) {
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, false);
}

int pa_decode_budget(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
                     const pa_bf16 *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, float scale, int max_ctas,
                     void *workspace, size_t workspace_bytes, void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, false, nullptr,
                      nullptr, false, nullptr, 0, max_ctas);
}

int quest_sparse_decode(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
                        const pa_bf16 *value_cache, const int32_t *block_tables,
                        int max_blocks_per_seq, const int32_t *context_lens,
                        const int32_t *selected, int topk, int batch, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                        float scale, void *workspace, size_t workspace_bytes, void *stream) {
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, selected, topk, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, true);
}

int quest_sparse_decode_budget(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
                               const pa_bf16 *value_cache, const int32_t *block_tables,
                               int max_blocks_per_seq, const int32_t *context_lens,
                               const int32_t *selected, int topk, int batch, int num_q_heads,
                               int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                               float scale, int max_ctas, void *workspace, size_t workspace_bytes,
                               void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, selected, topk, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, true, nullptr,
                      nullptr, false, nullptr, 0, max_ctas);
}

int quest_update_meta(pa_bf16 *kmin, pa_bf16 *kmax, const pa_bf16 *key,
                      const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!kmin || !kmax || !key || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!shape_supported(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(key)) return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_update_meta(kmin, kmax, key, slot_mapping, num_tokens, num_kv_heads,
                                             head_dim, block_size, num_blocks,
                                             static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_reshape_and_cache(const pa_bf16 *key, const pa_bf16 *value, pa_bf16 *key_cache,
                            pa_bf16 *value_cache, pa_bf16 *kmin, pa_bf16 *kmax,
                            const int64_t *slot_mapping, int64_t num_tokens, int num_kv_heads,
                            int head_dim, int block_size, int64_t num_blocks, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !kmin || !kmax || !slot_mapping)
        return PA_ERR_INVALID_ARG;
    if (!shape_supported(head_dim, block_size)) return PA_ERR_UNSUPPORTED;
    if (num_tokens > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        !aligned16(kmin) || !aligned16(kmax))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_write_quest(key_cache, value_cache, kmin, kmax, key, value,
                                             slot_mapping, num_tokens, num_kv_heads, head_dim,
                                             block_size, num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_rebuild_meta(pa_bf16 *kmin, pa_bf16 *kmax, const pa_bf16 *key_cache,
                       const int32_t *block_tables, int max_blocks_per_seq,
                       const int32_t *context_lens, int batch, int num_kv_heads, int head_dim,
                       int block_size, int64_t num_blocks, void *stream) {
    if (!kmin || !kmax || !key_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (batch <= 0 || max_blocks_per_seq <= 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (!shape_supported(head_dim, block_size) || batch > 65535) return PA_ERR_UNSUPPORTED;
    if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(key_cache)) return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_rebuild_meta(kmin, kmax, key_cache, block_tables,
                                              max_blocks_per_seq, context_lens, batch, num_kv_heads,
                                              head_dim, block_size, num_blocks,
                                              static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t quest_select_workspace_size(int batch, int num_kv_heads, int max_blocks_per_seq) {
    if (batch <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0) return 0;
    const size_t bytes = size_t(batch) * num_kv_heads * max_blocks_per_seq * sizeof(float);
    return (bytes + 255) / 256 * 256;
}

int quest_select_topk(int32_t *selected, const pa_bf16 *query, const pa_bf16 *kmin,
                      const pa_bf16 *kmax, const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, int topk, void *workspace,
                      size_t workspace_bytes, void *stream) {
    if (!selected || !query || !kmin || !kmax || !block_tables || !context_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0 || topk <= 0 || head_dim <= 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (!shape_supported(head_dim, block_size) || batch > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if (int64_t(max_blocks_per_seq) * block_size > int64_t(1) << 30) return PA_ERR_UNSUPPORTED;
    if (!aligned16(query) || !aligned16(kmin) || !aligned16(kmax) || !aligned16(workspace))
        return PA_ERR_INVALID_ARG;
    if (workspace_bytes < quest_select_workspace_size(batch, num_kv_heads, max_blocks_per_seq))
        return PA_ERR_WORKSPACE;
    const cudaError_t e = launch_quest_select(
        selected, static_cast<float *>(workspace), query, kmin, kmax, block_tables,
        max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size,
        num_blocks, topk, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

size_t quest_decode_workspace_size(int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int max_blocks_per_seq) {
    const size_t dec = pa_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim);
    const size_t sc = quest_select_workspace_size(batch, num_kv_heads, max_blocks_per_seq);
    if (dec == 0 || sc == 0) return 0;
    return (dec + 255) / 256 * 256 + sc;
}

namespace {
// score launch + fused top-K / sparse decode launch (bf16 or E4M3 cache)
int run_quest_decode(pa_bf16 *out, int32_t *selected, const pa_bf16 *query, const void *kmin,
                     const void *kmax, const void *key_cache, const void *value_cache,
                     const float *k_scale, const float *v_scale, const int32_t *block_tables, int MBS,
                     const int32_t *context_lens, int B, int Hq, int Hkv, int D, int BS, int64_t NB,
                     int topk, float scale, int max_ctas, void *workspace, size_t workspace_bytes,
                     void *stream, bool fp8, bool bscale = false, const ScoreWrite *sw = nullptr) {
    if (!selected || !kmin || !kmax || !workspace || max_ctas < 0) return PA_ERR_INVALID_ARG;
    int rc = check_attention_args(out, query, key_cache, value_cache, block_tables, MBS, context_lens, B, Hq,
                                  Hkv, D, BS, NB, scale, workspace);
    if (rc != PA_OK) return rc;
    if (topk <= 0) return PA_ERR_INVALID_ARG;
    if (fp8 && D != 128) return PA_ERR_UNSUPPORTED;
    if (!aligned16(kmin) || !aligned16(kmax)) return PA_ERR_INVALID_ARG;
    const size_t dec = pa_decode_workspace_size(B, Hq, Hkv, D);
    const size_t need = quest_decode_workspace_size(B, Hq, Hkv, D, MBS);
    if (dec == 0 || need == 0) return PA_ERR_UNSUPPORTED;
    if (workspace_bytes < need) return PA_ERR_WORKSPACE;
    float *scores = reinterpret_cast<float *>(static_cast<uint8_t *>(workspace) + (dec + 255) / 256 * 256);
    DecodeGeometry geo;
    cudaError_t e = decode_geometry(D, &geo, fp8);
    if (e != cudaSuccess) return cuda_fail(e);
    if (int64_t(B) * Hkv * topk >= int64_t(geo.grid) * kSparseLargeItems) {
        // A large selection: every CTA holds several whole segments, and their
        // top-Ks would run one after another inside it; the top-K kernel
        // (one CTA per segment) runs them all at once instead.
        e = launch_quest_select(selected, scores, query, kmin, kmax, block_tables, MBS, context_lens, B, Hq, Hkv,
                                D, BS, NB, topk, static_cast<cudaStream_t>(stream), fp8, bscale ? k_scale : nullptr,
                                sw);
        if (e != cudaSuccess) return cuda_fail(e);
        return run_decode(out, query, key_cache, value_cache, block_tables, MBS, context_lens, selected, topk, B,
                          Hq, Hkv, D, BS, NB, scale, workspace, dec, stream, true, k_scale, v_scale, fp8, nullptr,
                          0, max_ctas, nullptr, nullptr, bscale);
    }
    e = launch_quest_scores(scores, query, kmin, kmax, block_tables, MBS, context_lens, B, Hq, Hkv, D, BS, NB,
                            static_cast<cudaStream_t>(stream), fp8, bscale ? k_scale : nullptr, sw);
    if (e != cudaSuccess) return cuda_fail(e);
    return run_decode(out, query, key_cache, value_cache, block_tables, MBS, context_lens, nullptr, topk, B,
                      Hq, Hkv, D, BS, NB, scale, workspace, dec, stream, true, k_scale, v_scale, fp8, nullptr, 0,
                      max_ctas, scores, selected, bscale);
}
}  // namespace

int quest_decode(pa_bf16 *out, int32_t *selected, const pa_bf16 *query, const pa_bf16 *kmin,
                 const pa_bf16 *kmax, const pa_bf16 *key_cache, const pa_bf16 *value_cache,
                 const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                 int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                 int64_t num_blocks, int topk, float scale, int max_ctas, void *workspace,
                 size_t workspace_bytes, void *stream) {
    return run_quest_decode(out, selected, query, kmin, kmax, key_cache, value_cache, nullptr, nullptr,
                            block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, topk, scale, max_ctas, workspace, workspace_bytes,
                            stream, false);
}

int quest_decode_fp8(pa_bf16 *out, int32_t *selected, const pa_bf16 *query, const pa_e4m3 *kmin,
                     const pa_e4m3 *kmax, const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                     const float *k_scale, const float *v_scale, const int32_t *block_tables,
                     int max_blocks_per_seq, const int32_t *context_lens, int batch, int num_q_heads,
                     int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int topk,
                     float scale, int max_ctas, void *workspace, size_t workspace_bytes, void *stream) {
    if (!k_scale || !v_scale) return PA_ERR_INVALID_ARG;
    return run_quest_decode(out, selected, query, kmin, kmax, key_cache, value_cache, k_scale, v_scale,
                            block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, topk, scale, max_ctas, workspace, workspace_bytes,
                            stream, true);
}

/* ----------------------------------- the step's write folded into decode */

namespace {
int check_step_write(const pa_bf16 *key, const pa_bf16 *value, const int64_t *slot_mapping, int batch) {
    if (!key || !value || !slot_mapping || batch <= 0) return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value)) return PA_ERR_INVALID_ARG;
    return PA_OK;
}
}  // namespace

int pa_reshape_and_decode(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key, const pa_bf16 *value,
                          const int64_t *slot_mapping, pa_bf16 *key_cache, pa_bf16 *value_cache, pa_bf16 *kmin,
                          pa_bf16 *kmax, const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, float scale, void *workspace,
                          size_t workspace_bytes, void *stream) {
    int rc = check_step_write(key, value, slot_mapping, batch);
    if (rc != PA_OK) return rc;
    if ((kmin == nullptr) != (kmax == nullptr)) return PA_ERR_INVALID_ARG;
    if (kmin && (!aligned16(kmin) || !aligned16(kmax))) return PA_ERR_INVALID_ARG;
    const ScoreWrite sw{key, value, slot_mapping, key_cache, value_cache, kmin, kmax};
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens, nullptr,
                      0, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, workspace,
                      workspace_bytes, stream, false, nullptr, nullptr, false, nullptr, 0, 0, nullptr, nullptr,
                      false, &sw);
}

int quest_reshape_and_decode(pa_bf16 *out, int32_t *selected, const pa_bf16 *query, const pa_bf16 *key,
                             const pa_bf16 *value, const int64_t *slot_mapping, pa_bf16 *kmin, pa_bf16 *kmax,
                             pa_bf16 *key_cache, pa_bf16 *value_cache, const int32_t *block_tables,
                             int max_blocks_per_seq, const int32_t *context_lens, int batch, int num_q_heads,
                             int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int topk,
                             float scale, int max_ctas, void *workspace, size_t workspace_bytes, void *stream) {
    int rc = check_step_write(key, value, slot_mapping, batch);
    if (rc != PA_OK) return rc;
    const ScoreWrite sw{key, value, slot_mapping, key_cache, value_cache, kmin, kmax};
    return run_quest_decode(out, selected, query, kmin, kmax, key_cache, value_cache, nullptr, nullptr,
                            block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, topk, scale, max_ctas, workspace, workspace_bytes,
                            stream, false, false, &sw);
}

int pa_workspace_status(const void *workspace, void *stream) {
    if (!workspace) return PA_ERR_INVALID_ARG;
    int32_t st = 0;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&st, workspace, sizeof st, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e);
    return st == 0 ? PA_OK : PA_ERR_DEVICE;
}

int pa_check_metadata(int32_t *counts, const int64_t *slot_mapping, int64_t num_tokens,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *context_lens, int batch, int block_size, int64_t num_blocks,
                      void *stream) {
    if (!counts || num_tokens < 0 || batch < 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_tokens > 0 && !slot_mapping) return PA_ERR_INVALID_ARG;
    if (block_tables && (!context_lens || max_blocks_per_seq <= 0)) return PA_ERR_INVALID_ARG;
    if (num_tokens > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    const cudaError_t e = launch_check_metadata(counts, slot_mapping, num_tokens, block_tables,
                                                max_blocks_per_seq, context_lens, batch, block_size,
                                                num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"

/* ------------------------------------------------- 8-bit (E4M3) KV cache */

namespace {
// shared checks of the fp8 write / metadata entry points
int check_fp8_write(int64_t num_tokens, int num_kv_heads, int head_dim, int block_size,
                    int64_t num_blocks) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 128 || block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
    if (num_tokens > (int64_t(1) << 31) - 1) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}
}  // namespace

extern "C" {

int pa_reshape_and_cache_fp8(const pa_bf16 *key, const pa_bf16 *value, pa_e4m3 *key_cache,
                             pa_e4m3 *value_cache, const int64_t *slot_mapping, int64_t num_tokens,
                             const float *k_scale, const float *v_scale, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, void *stream) {
    int rc = check_fp8_write(num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping || !k_scale || !v_scale)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_write_fp8(key_cache, value_cache, nullptr, nullptr, key, value, k_scale,
                                           v_scale, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                           block_size, num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_reshape_and_cache_fp8(const pa_bf16 *key, const pa_bf16 *value, pa_e4m3 *key_cache,
                                pa_e4m3 *value_cache, pa_e4m3 *kmin, pa_e4m3 *kmax,
                                const int64_t *slot_mapping, int64_t num_tokens, const float *k_scale,
                                const float *v_scale, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, void *stream) {
    int rc = check_fp8_write(num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !kmin || !kmax || !slot_mapping || !k_scale ||
        !v_scale)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        !aligned16(kmin) || !aligned16(kmax))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_write_fp8(key_cache, value_cache, kmin, kmax, key, value, k_scale, v_scale,
                                           slot_mapping, num_tokens, num_kv_heads, head_dim, block_size,
                                           num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_update_meta_fp8(pa_e4m3 *kmin, pa_e4m3 *kmax, const pa_bf16 *key, const int64_t *slot_mapping,
                          int64_t num_tokens, const float *k_scale, int num_kv_heads, int head_dim,
                          int block_size, int64_t num_blocks, void *stream) {
    int rc = check_fp8_write(num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!kmin || !kmax || !key || !slot_mapping || !k_scale) return PA_ERR_INVALID_ARG;
    if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(key)) return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_update_meta_fp8(kmin, kmax, key, k_scale, slot_mapping, num_tokens,
                                                 num_kv_heads, head_dim, block_size, num_blocks,
                                                 static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_rebuild_meta_fp8(pa_e4m3 *kmin, pa_e4m3 *kmax, const pa_e4m3 *key_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *context_lens, int batch, int num_kv_heads, int head_dim,
                           int block_size, int64_t num_blocks, void *stream) {
    if (!kmin || !kmax || !key_cache || !block_tables || !context_lens) return PA_ERR_INVALID_ARG;
    if (batch <= 0 || max_blocks_per_seq <= 0 || num_kv_heads <= 0 || num_blocks <= 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != 128 || block_size != kBlockSize || batch > 65535) return PA_ERR_UNSUPPORTED;
    if (!aligned16(kmin) || !aligned16(kmax) || !aligned16(key_cache)) return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_rebuild_meta_fp8(kmin, kmax, key_cache, block_tables, max_blocks_per_seq,
                                                  context_lens, batch, num_kv_heads, head_dim, block_size,
                                                  num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

}  // extern "C"

namespace {
int run_select_fp8(int32_t *selected, const pa_bf16 *query, const pa_e4m3 *kmin, const pa_e4m3 *kmax,
                   const float *k_bscale, const int32_t *block_tables, int max_blocks_per_seq,
                   const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads, int head_dim,
                   int block_size, int64_t num_blocks, int topk, void *workspace, size_t workspace_bytes,
                   void *stream) {
    if (!selected || !query || !kmin || !kmax || !block_tables || !context_lens || !workspace)
        return PA_ERR_INVALID_ARG;
    if (batch <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || max_blocks_per_seq <= 0 ||
        num_blocks <= 0 || topk <= 0 || head_dim <= 0 || block_size <= 0)
        return PA_ERR_INVALID_ARG;
    if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
    if (head_dim != 128 || block_size != kBlockSize || batch > kMaxBatch) return PA_ERR_UNSUPPORTED;
    if (int64_t(max_blocks_per_seq) * block_size > int64_t(1) << 30) return PA_ERR_UNSUPPORTED;
    if (!aligned16(query) || !aligned16(kmin) || !aligned16(kmax) || !aligned16(workspace))
        return PA_ERR_INVALID_ARG;
    if (workspace_bytes < quest_select_workspace_size(batch, num_kv_heads, max_blocks_per_seq))
        return PA_ERR_WORKSPACE;
    const cudaError_t e = launch_quest_select(
        selected, static_cast<float *>(workspace), query, kmin, kmax, block_tables, max_blocks_per_seq,
        context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, topk,
        static_cast<cudaStream_t>(stream), true, k_bscale);
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}
}  // namespace

extern "C" {

int quest_select_topk_fp8(int32_t *selected, const pa_bf16 *query, const pa_e4m3 *kmin,
                          const pa_e4m3 *kmax, const int32_t *block_tables, int max_blocks_per_seq,
                          const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                          int head_dim, int block_size, int64_t num_blocks, int topk, void *workspace,
                          size_t workspace_bytes, void *stream) {
    return run_select_fp8(selected, query, kmin, kmax, nullptr, block_tables, max_blocks_per_seq, context_lens,
                          batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, topk, workspace,
                          workspace_bytes, stream);
}

/* ------------------------------------ E4M3 cache with per-block scales */

int pa_reshape_and_cache_fp8_block(const pa_bf16 *key, const pa_bf16 *value, pa_e4m3 *key_cache,
                                   pa_e4m3 *value_cache, const int64_t *slot_mapping, int64_t num_tokens,
                                   float *k_bscale, float *v_bscale, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, void *stream) {
    int rc = check_fp8_write(num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !slot_mapping || !k_bscale || !v_bscale)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_write_fp8_block(key_cache, value_cache, nullptr, nullptr, k_bscale, v_bscale,
                                                 key, value, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                                 block_size, num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_reshape_and_cache_fp8_block(const pa_bf16 *key, const pa_bf16 *value, pa_e4m3 *key_cache,
                                      pa_e4m3 *value_cache, pa_e4m3 *kmin, pa_e4m3 *kmax,
                                      const int64_t *slot_mapping, int64_t num_tokens, float *k_bscale,
                                      float *v_bscale, int num_kv_heads, int head_dim, int block_size,
                                      int64_t num_blocks, void *stream) {
    int rc = check_fp8_write(num_tokens, num_kv_heads, head_dim, block_size, num_blocks);
    if (rc != PA_OK) return rc;
    if (num_tokens == 0) return PA_OK;
    if (!key || !value || !key_cache || !value_cache || !kmin || !kmax || !slot_mapping || !k_bscale ||
        !v_bscale)
        return PA_ERR_INVALID_ARG;
    if (!aligned16(key) || !aligned16(value) || !aligned16(key_cache) || !aligned16(value_cache) ||
        !aligned16(kmin) || !aligned16(kmax))
        return PA_ERR_INVALID_ARG;
    const cudaError_t e = launch_write_fp8_block(key_cache, value_cache, kmin, kmax, k_bscale, v_bscale, key,
                                                 value, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                                 block_size, num_blocks, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : cuda_fail(e);
}

int quest_select_topk_fp8_block(int32_t *selected, const pa_bf16 *query, const pa_e4m3 *kmin,
                                const pa_e4m3 *kmax, const float *k_bscale, const int32_t *block_tables,
                                int max_blocks_per_seq, const int32_t *context_lens, int batch,
                                int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                int64_t num_blocks, int topk, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if (!k_bscale) return PA_ERR_INVALID_ARG;
    return run_select_fp8(selected, query, kmin, kmax, k_bscale, block_tables, max_blocks_per_seq, context_lens,
                          batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, topk, workspace,
                          workspace_bytes, stream);
}

int pa_decode_fp8_block(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                        const pa_e4m3 *value_cache, const float *k_bscale, const float *v_bscale,
                        const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                        int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                        void *stream) {
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                      nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                      workspace, workspace_bytes, stream, false, k_bscale, v_bscale, true, nullptr, 0, 0,
                      nullptr, nullptr, true);
}

int pa_decode_fp8_block_budget(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                               const pa_e4m3 *value_cache, const float *k_bscale, const float *v_bscale,
                               const int32_t *block_tables, int max_blocks_per_seq,
                               const int32_t *context_lens, int batch, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int64_t num_blocks, float scale, int max_ctas,
                               void *workspace, size_t workspace_bytes, void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                      nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                      workspace, workspace_bytes, stream, false, k_bscale, v_bscale, true, nullptr, 0, max_ctas,
                      nullptr, nullptr, true);
}

int quest_sparse_decode_fp8_block(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                                  const pa_e4m3 *value_cache, const float *k_bscale, const float *v_bscale,
                                  const int32_t *block_tables, int max_blocks_per_seq,
                                  const int32_t *context_lens, const int32_t *selected, int topk, int batch,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, float scale, int max_ctas, void *workspace,
                                  size_t workspace_bytes, void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                      selected, topk, batch, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                      workspace, workspace_bytes, stream, true, k_bscale, v_bscale, true, nullptr, 0, max_ctas,
                      nullptr, nullptr, true);
}

int quest_decode_fp8_block(pa_bf16 *out, int32_t *selected, const pa_bf16 *query, const pa_e4m3 *kmin,
                           const pa_e4m3 *kmax, const pa_e4m3 *key_cache, const pa_e4m3 *value_cache,
                           const float *k_bscale, const float *v_bscale, const int32_t *block_tables,
                           int max_blocks_per_seq, const int32_t *context_lens, int batch, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks, int topk,
                           float scale, int max_ctas, void *workspace, size_t workspace_bytes, void *stream) {
    if (!k_bscale || !v_bscale) return PA_ERR_INVALID_ARG;
    return run_quest_decode(out, selected, query, kmin, kmax, key_cache, value_cache, k_bscale, v_bscale,
                            block_tables, max_blocks_per_seq, context_lens, batch, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, topk, scale, max_ctas, workspace, workspace_bytes,
                            stream, true, true);
}

int quest_sparse_decode_fp8_budget(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                                   const pa_e4m3 *value_cache, const float *k_scale, const float *v_scale,
                                   const int32_t *block_tables, int max_blocks_per_seq,
                                   const int32_t *context_lens, const int32_t *selected, int topk,
                                   int batch, int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int64_t num_blocks, float scale, int max_ctas,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, selected, topk, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, true, k_scale,
                      v_scale, true, nullptr, 0, max_ctas);
}

int pa_decode_fp8(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                  const pa_e4m3 *value_cache, const float *k_scale, const float *v_scale,
                  const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                  int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                  void *stream) {
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, false, k_scale,
                      v_scale, true);
}

int pa_decode_fp8_budget(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                         const pa_e4m3 *value_cache, const float *k_scale, const float *v_scale,
                         const int32_t *block_tables, int max_blocks_per_seq, const int32_t *context_lens,
                         int batch, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                         int64_t num_blocks, float scale, int max_ctas, void *workspace,
                         size_t workspace_bytes, void *stream) {
    if (max_ctas < 0) return PA_ERR_INVALID_ARG;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, nullptr, 0, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, false, k_scale,
                      v_scale, true, nullptr, 0, max_ctas);
}

int quest_sparse_decode_fp8(pa_bf16 *out, const pa_bf16 *query, const pa_e4m3 *key_cache,
                            const pa_e4m3 *value_cache, const float *k_scale, const float *v_scale,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *context_lens, const int32_t *selected, int topk, int batch,
                            int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                            int64_t num_blocks, float scale, void *workspace, size_t workspace_bytes,
                            void *stream) {
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                      context_lens, selected, topk, batch, num_q_heads, num_kv_heads, head_dim,
                      block_size, num_blocks, scale, workspace, workspace_bytes, stream, true, k_scale,
                      v_scale, true);
}

}  // extern "C"

extern "C" {

size_t pa_decode_multi_workspace_size(int total_q, int num_q_heads, int num_kv_heads, int head_dim) {
    if (total_q <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads != 0) return 0;
    if (total_q > kMaxMultiRows || !shape_supported(head_dim, kBlockSize)) return 0;
    DecodeGeometry geo;
    if (decode_geometry(head_dim, &geo) != cudaSuccess) return 0;
    return decode_multi_workspace_bytes(total_q, num_kv_heads, head_dim, geo.workers);
}

int pa_decode_multi(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
                    const pa_bf16 *value_cache, const int32_t *block_tables, int max_blocks_per_seq,
                    const int32_t *cu_seqlens_q, const int32_t *context_lens, int batch, int total_q,
                    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                    float scale, void *workspace, size_t workspace_bytes, void *stream) {
    if (batch <= 0 || total_q < 0 || !cu_seqlens_q) return PA_ERR_INVALID_ARG;
    if (batch > kMaxMultiRows || total_q > kMaxMultiRows) return PA_ERR_UNSUPPORTED;
    if (total_q == 0) return PA_OK;
    return run_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq, context_lens,
                      nullptr, 0, total_q, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
                      scale, workspace, workspace_bytes, stream, false, nullptr, nullptr, false,
                      cu_seqlens_q, batch);
}

}  // extern "C"

#ifdef PA_FAULT_TEST
// Failure-test build only: every later decode launch gives up a bounded wait
// after wait_ns (0: the default 0.5 s) and its producer stops issuing at item
// stop_item of each CTA's range (negative: never), so the consumers' waits
// for the stages that are never armed run out.
extern "C" PA_API void pa_fault_test_configure(int stop_item, uint64_t wait_ns) {
    g_wait_ns.store(wait_ns ? wait_ns : kDefaultWaitNs, std::memory_order_relaxed);
    g_stop_item.store(stop_item < 0 ? INT_MAX : stop_item, std::memory_order_relaxed);
}
#endif
