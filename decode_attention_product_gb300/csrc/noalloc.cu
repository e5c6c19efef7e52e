// noalloc.cu -- aq_decode_attention_noalloc: PQ decode attention that needs no
// workspace from the caller.
//
// aq_decode_attention asks its caller for device scratch when it splits long
// sequences (one (max, sum, output) partial per request, query head and
// split).  Some callers have no way to provide that: a plugin or operator that
// is handed only the tensors of the call and must not touch the host
// framework's memory pool, a process whose device memory is entirely reserved
// by another allocator, or a latency-critical loop in which an allocation (which
// can synchronise the device and can fail) is not allowed.  This entry point
// keeps the partials in one fixed array that the library owns instead.
//
// The array is a file-scope __device__ variable of kScratchBytes (4 MiB): every
// GPU on which the library's code is loaded holds it until the process exits.
// In host code its name is only a stand-in, so its device address is looked up
// with cudaGetSymbolAddress, once per device, on the first call made while that
// device is current; that first call should therefore come before any stream
// capture.  The address is kept until the process exits: a cudaDeviceReset of
// the device invalidates it, and the entry point is not to be called on that
// device afterwards.  All calls share the one array and nothing in it is kept for the
// caller: every partial is written by the split kernel before the combine
// kernel reads it, so it needs no clearing, but two calls whose kernels overlap
// on the GPU (different streams or host threads) race on it.
#include <cstdio>
#include <mutex>

#include "aqpq.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(4) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

std::mutex g_mu;
void *g_scratch_addr[kMaxDevices] = {};

}  // namespace

extern "C" aq_status aq_decode_attention_noalloc(
    const aq_pq_config *cfg, int32_t batch, int32_t num_q_heads, int32_t num_kv_heads, const float *q,
    const uint8_t *code_pages, int64_t num_pages, const void *codebooks_f16, int64_t num_sets,
    const int32_t *req_set, const int32_t *block_table, int32_t max_pages, const int32_t *seq_lens,
    int32_t max_seq_len, float scale, int32_t num_splits, float *out, int32_t *device_status,
    aq_stream_t stream) {
    // the scratch this call would need (host arithmetic only)
    size_t need = 0;
    aq_status st = aq_decode_plan(cfg, batch, num_q_heads, num_kv_heads, max_seq_len, num_splits, 0,
                                  nullptr, nullptr, &need);
    if (st != AQ_OK) return st;
    if (need > kScratchBytes) return AQ_ERR_WORKSPACE_TOO_SMALL;
    void *scratch = nullptr;
    if (need > 0 && batch > 0) {
        int dev = -1;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) {
            aq::record_cuda_error(e);
            return AQ_ERR_CUDA;
        }
        if (dev < 0 || dev >= kMaxDevices) return AQ_ERR_UNSUPPORTED;
        std::lock_guard<std::mutex> lock(g_mu);
        if (!g_scratch_addr[dev]) {
            void *addr = nullptr;
            e = cudaGetSymbolAddress(&addr, g_noalloc_scratch);
            if (e != cudaSuccess || addr == nullptr) {
                aq::record_cuda_error(e != cudaSuccess ? e : cudaErrorInvalidSymbol);
                return AQ_ERR_CUDA;
            }
            g_scratch_addr[dev] = addr;
        }
        scratch = g_scratch_addr[dev];
    }
    return aq_decode_attention(cfg, batch, num_q_heads, num_kv_heads, q, code_pages, num_pages,
                               codebooks_f16, num_sets, req_set, block_table, max_pages, seq_lens,
                               max_seq_len, scale, num_splits, out, scratch, kScratchBytes,
                               device_status, stream);
}
