// no_alloc.cu -- pa_decode_no_alloc: dense paged decode attention whose
// scratch lives in a fixed buffer compiled into the library.
//
// Who needs this: a caller that may not allocate device memory at all, for
// example a plugin inside a serving engine that hands it only the tensors it
// owns (query, caches, tables, output) and keeps every other byte of HBM for
// its own KV-cache pool, or a latency-critical loop where cudaMalloc and
// cudaFree are off limits because they can synchronise the device. Such a
// caller cannot provide the workspace pa_decode asks for.
//
// The scratch (status word, per-sequence arrival counters, split-KV partial
// outputs) is one file-scope __device__ array of kNoAllocScratchBytes. Every
// GPU that loads the library carries it until the process exits. In host code
// the array's name is only a host-side stand-in, so the entry point looks up
// its device address once per device with cudaGetSymbolAddress, on that
// device, during its first call there; make that first call before any
// stream capture. All calls share the one array: the status word and the
// counters are cleared on the caller's stream at the start of every call, and
// calls that overlap in time on the GPU (different streams, or different host
// threads) race on it.
#include <mutex>

#include "../../include/paged_decode.h"
#include "kernels.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(PA_NO_ALLOC_SCRATCH_BYTES);

static __device__ __align__(256) unsigned char g_no_alloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices];
std::mutex g_scratch_mu;

}  // namespace

extern "C" int pa_decode_no_alloc(pa_bf16 *out, const pa_bf16 *query, const pa_bf16 *key_cache,
                                  const pa_bf16 *value_cache, const int32_t *block_tables,
                                  int max_blocks_per_seq, const int32_t *context_lens, int batch,
                                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                                  int64_t num_blocks, float scale, void *stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        if (!g_scratch_ptr[dev]) {
            void *p = nullptr;
            e = cudaGetSymbolAddress(&p, g_no_alloc_scratch);
            if (e != cudaSuccess || !p) return PA_ERR_CUDA;
            g_scratch_ptr[dev] = p;
        }
        scratch = g_scratch_ptr[dev];
    }
    const size_t need = pa_decode_workspace_size(batch, num_q_heads, num_kv_heads, head_dim);
    if (need == 0)  // invalid or unsupported shape: let pa_decode name the error
        return pa_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                         context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                         num_blocks, scale, scratch, 0, stream);
    if (need > kNoAllocScratchBytes) return PA_ERR_WORKSPACE;  // problem too large for the buffer
    // status word (256 B) and one arrival counter per (sequence, KV head) must
    // start at zero; the previous call may have left them set if it gave up
    const size_t counters = (size_t(batch) * size_t(num_kv_heads) * 4 + 255) / 256 * 256;
    e = cudaMemsetAsync(scratch, 0, 256 + counters, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode(out, query, key_cache, value_cache, block_tables, max_blocks_per_seq,
                     context_lens, batch, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, scratch, kNoAllocScratchBytes, stream);
}

extern "C" int pa_decode_no_alloc_status(void *stream) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_scratch_mu);
        scratch = g_scratch_ptr[dev];
    }
    if (!scratch) return PA_ERR_INVALID_ARG;  // no call on this device yet
    return pa_workspace_status(scratch, stream);
}
