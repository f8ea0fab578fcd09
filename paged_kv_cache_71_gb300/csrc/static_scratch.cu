// static_scratch.cu -- paged decode attention for callers that cannot allocate.
//
// Some callers cannot call cudaMalloc (or any allocator) at the point where
// they run attention: code that must not allocate once its memory budget is
// fixed, plugin hosts that own every device allocation, or runtimes whose
// allocator is not reachable from the C ABI.  For them this file keeps the
// split-KV scratch (completion counters and partial (m, l, O) records) in a
// fixed, file-scope device array instead of a caller-provided workspace.
//
// The array costs PKV_STATIC_SCRATCH_BYTES of device memory on every GPU that
// loads the library, for as long as the process lives.  Every call shares
// it: its counters are cleared by each call, its partial records are
// overwritten, and two calls whose work overlaps on the GPU (other streams,
// other host threads) race on it.
#include <mutex>

#include "pkv_device.cuh"

#define PKV_API extern "C" __attribute__((visibility("default")))

namespace pkv {
void set_last_error(const char* msg);  // api.cu
}

namespace {

constexpr size_t kStaticScratchBytes = PKV_STATIC_SCRATCH_BYTES;

static __device__ __align__(256) uint8_t g_static_scratch[kStaticScratchBytes];

constexpr int kMaxDevices = 64;
static void* g_scratch_addr[kMaxDevices];
static std::mutex g_scratch_mu;

// Device address of g_static_scratch on the current device, looked up once
// per device (the host-side name of the array is not a device address).
static pkv_status scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return PKV_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return PKV_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess || p == nullptr) {
            pkv::set_last_error("cudaGetSymbolAddress of the static scratch array failed");
            return PKV_ERR_CUDA;
        }
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return PKV_OK;
}

}  // namespace

PKV_API pkv_status pkv_paged_attention_decode_static_scratch(
    void* out, const void* q, int32_t q_dtype, const void* k_cache, const void* v_cache, const pkv_cache_desc* cache,
    const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens, int32_t num_seqs,
    int32_t num_q_heads, float scale, int32_t num_splits, int32_t max_context_len, int32_t* device_error,
    void* stream) {
    size_t need = 0;
    pkv_status st = pkv_paged_attention_workspace_size(cache, num_seqs, num_q_heads, num_splits, &need);
    if (st != PKV_OK) return st;
    if (need > kStaticScratchBytes) {
        pkv::set_last_error("static scratch of PKV_STATIC_SCRATCH_BYTES is too small for this batch; "
                            "use pkv_paged_attention_decode with a caller workspace, or num_splits = 1");
        return PKV_ERR_WORKSPACE;
    }
    void* scratch = nullptr;
    if (need > 0) {
        st = scratch_address(&scratch);
        if (st != PKV_OK) return st;
    }
    return pkv_paged_attention_decode(out, q, q_dtype, k_cache, v_cache, cache, block_tables, max_blocks_per_seq,
                                      context_lens, num_seqs, num_q_heads, scale, num_splits, max_context_len,
                                      scratch, need > 0 ? kStaticScratchBytes : 0, device_error, stream);
}
