// attn_decode_paged_noalloc: paged decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc (or any allocating routine) on their decode path:
// for example a plug-in inside a host application that owns the whole device-memory
// budget through its own pool, or a latency-critical token loop where cudaMalloc's
// implicit device synchronisation would stall every other stream. For them this entry
// point takes the decode kernel's scratch (split partials and per-request offsets into
// them) from a fixed buffer compiled into the library instead of from a workspace.
//
// The buffer is a file-scope __device__ array of kScratchBytes (16 MiB). Every GPU that
// loads this part of the library holds it until the process exits. In host code the
// array's name only stands for the device symbol; its device address is looked up once
// per device (cudaGetSymbolAddress, with that device current) on the first call made
// while that device is current, and cached.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/attn.h"
#include "attn_internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(16) << 20;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[kScratchBytes];

std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};


// Device address of the scratch array on the current device (looked up once per device).
void* scratch_for_current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace

extern "C" {

ATTN_API size_t attn_decode_paged_noalloc_max_bytes(void) { return kScratchBytes; }

ATTN_API int attn_decode_paged_noalloc(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                                       const int32_t* block_table, const int32_t* seq_lens, attn_bf16* o, float* lse,
                                       int B, int Hq, int Hkv, int D, int page_size, int max_pages_per_seq,
                                       int num_pages, float scale, int window, void* stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || D <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (D != 128 && D != 256) return ATTN_ERR_UNSUPPORTED;  // before sizing: no other head size has a size
    const size_t need = attn_workspace_size(ATTN_OP_DECODE_PAGED, B, Hq, Hkv, 0, D, 0, max_pages_per_seq);
    if (need > kScratchBytes) return ATTN_ERR_WORKSPACE;  // beyond the built-in buffer
    if (B == 0) return attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, D, page_size,
                                         max_pages_per_seq, num_pages, scale, window, nullptr, 0, stream);
    void* scratch = scratch_for_current_device();
    if (!scratch) return ATTN_ERR_NO_DEVICE;
    return attn_decode_paged(q, k_cache, v_cache, block_table, seq_lens, o, lse, B, Hq, Hkv, D, page_size,
                             max_pages_per_seq, num_pages, scale, window, scratch, kScratchBytes, stream);
}

}  // extern "C"
