// C ABI of the attention library (declared in include/attn.h): argument checks,
// workspace layout, TMA tensor maps and kernel launches. No allocation, no host
// synchronisation except in attn_get_device_status().
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <map>
#include <mutex>
#include <string>
#include <vector>

#include "../../include/attn.h"
#include "attn_internal.h"
#include "ptx.cuh"

namespace {

// [0]: fault flags; [1]: id of the first pipeline wait that gave up (0 = none).
__device__ unsigned g_attn_status[2] = {0u, 0u};

// One bounded pipeline wait that nothing completes: the wait gives up after limit_ns, records
// the timeout in the status word and the kernel returns (see attn_selftest_wait_timeout).
__global__ void selftest_wait_kernel(unsigned* status, unsigned long long limit_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        attn::mbar_init(attn::smem_u32(&bar), 1);
        abort_flag = 0;
        attn::fence_mbar_init();
        attn::mbar_wait_for(attn::smem_u32(&bar), 0, &abort_flag, status, 0x7f, limit_ns);
    }
}

constexpr int kMaxDevices = 64;

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

struct DeviceInfo {
    bool init = false;
    bool ok = false;
    int sms = 0;
    unsigned* status = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
EncodeTiledFn g_encode = nullptr;

// Per-device facts, queried once: sm_103, SM count, address of the status word.
const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        d.init = true;
        int major = 0, minor = 0;
        cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
        cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        void* p = nullptr;
        const bool sym = cudaGetSymbolAddress(&p, g_attn_status) == cudaSuccess;
        d.status = static_cast<unsigned*>(p);
        d.ok = major == 10 && minor == 3 && sym && d.sms > 0;
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                    cudaSuccess &&
                q == cudaDriverEntryPointSuccess)
                g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        if (!g_encode) d.ok = false;
    }
    return d.ok ? &d : nullptr;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 4-D map over a [batch, rows, heads, dim] bf16 tensor, box = 64 dims x 1 head x box_rows rows.
bool make_map(CUtensorMap* m, const void* base, int D, int H, int rows, int batch, int box_rows = 128) {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)rows * H * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D map over the fp32 dQ accumulator [batch, rows, heads, dim], box = 32 floats x 1 x 128 rows.
bool make_map_f32(CUtensorMap* m, const void* base, int D, int H, int rows, int batch) {
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)batch};
    cuuint64_t strides[3] = {(cuuint64_t)D * 4, (cuuint64_t)H * D * 4, (cuuint64_t)rows * H * D * 4};
    cuuint32_t box[4] = {32, 1, 128, 1};
    cuuint32_t es[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map over a paged cache [num_pages, 16, heads, dim] viewed as (64 dims, 8 rows, heads*dim/64
// chunks of 64 dims, 2 groups of 8 rows, pages); box = 64 x 8 x 2 x 2 x 1: 16 rows x 128 dims of
// one head of one page (4 KB), the two 64-dim chunks interleaved per 8-row group (D = 64: one
// chunk, 2 KB).
bool make_cache_map(CUtensorMap* m, const void* base, int D, int H, int num_pages, int chunks = 0) {
    const cuuint64_t row = (cuuint64_t)H * D * 2;
    cuuint64_t dims[5] = {64, 8, (cuuint64_t)H * D / 64, 2, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {row, 128, 8 * row, 16 * row};
    // the forward's slot width, 128 (or 64) dims; a CTA pair's K slot takes 256 (chunks = 4)
    cuuint32_t box[5] = {64, 8, chunks > 0 ? (cuuint32_t)chunks : D >= 128 ? 2u : 1u, 2, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int check_common(int Hq, int Hkv, float scale, int causal, int window) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    if (window < 0) return ATTN_ERR_INVALID_ARG;
    if (causal != 1) return ATTN_ERR_UNSUPPORTED;
    return ATTN_OK;
}

int check_prefill_shape(long long rows, int Hq, int Hkv, int D, int S) {
    if (D != 64 && D != 128 && D != 256 && D != 512) return ATTN_ERR_UNSUPPORTED;
    if (S > 65535LL * 128) return ATTN_ERR_UNSUPPORTED;
    if (rows > 0x7fffffffLL) return ATTN_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    (void)Hq, (void)Hkv;
    return ATTN_OK;
}

// CTAs per query tile and head in the forward: one per 256 output columns.
int fwd_splits(int D) { return D > 256 ? D / 256 : 1; }

size_t bwd_ws(long long rows, int Hq, int D) {
    return align256((size_t)rows * Hq * D * 4) + align256((size_t)rows * Hq * 4);
}

// CTAs per KV-head block of a decode launch at most: the blocks share decode_max_grid() CTAs.
int decode_grid_cap(int nhb) { return attn::decode_max_grid() / nhb > 1 ? attn::decode_max_grid() / nhb : 1; }

// Decode workspace: the split partials (slot (b + k) * 2 + half for CTA k of a head block, every
// head block writing only its own heads). Every call writes all of it that it reads: contents on
// entry do not matter.
// Returns 0 for a problem the decode kernels do not take (its call is rejected before any use).
bool decode_shape_ok(int Hq, int Hkv, int D) {
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return false;
    const int G = Hq / Hkv;
    return D == 128 ? (G == 1 || G == 2 || G == 4 || G == 8) : D == 256 ? (G == 1 || G == 2 || G == 4) : false;
}
size_t decode_ws(int B, int Hq, int Hkv, int D) {
    if (B < 0 || !decode_shape_ok(Hq, Hkv, D)) return 0;
    const int nhb = Hkv / attn::decode_heads_per_unit(Hkv, D, Hq / Hkv);
    return align256((size_t)(B + decode_grid_cap(nhb)) * 2 * Hq * attn::decode_row_floats(D) * 4);
}

// 3-D map over a paged cache [num_pages * 16 tokens, heads, dim]: box = dim x hb heads x 16 tokens,
// no swizzle, so one box lands as the [16][hb][dim] block the decode kernel reads.
bool make_decode_map(CUtensorMap* m, const void* base, int D, int H, int num_pages, int hb) {
    cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)num_pages * 16};
    cuuint64_t strides[2] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2};
    cuuint32_t box[3] = {(cuuint32_t)D, (cuuint32_t)hb, 16};
    cuuint32_t es[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map over a paged K or V cache [num_pages, 16, heads, D = 128] viewed as (64 dims, 16 tokens,
// heads, 2 halves of D, pages); box = 64 x 16 x hb x 2 x 1, the whole page of hb heads. Shared memory
// gets [half][head][token][64 dims], each token's 128-byte row swizzled by token % 8.
bool make_decode_swz_map(CUtensorMap* m, const void* base, int D, int H, int num_pages, int hb) {
    const cuuint64_t row = (cuuint64_t)H * D * 2;
    cuuint64_t dims[5] = {64, 16, (cuuint64_t)H, (cuuint64_t)D / 64, (cuuint64_t)num_pages};
    cuuint64_t strides[4] = {row, (cuuint64_t)D * 2, 128, 16 * row};
    cuuint32_t box[5] = {64, 16, (cuuint32_t)hb, (cuuint32_t)D / 64, 1};
    cuuint32_t es[5] = {1, 1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, const_cast<void*>(base), dims, strides, box, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int fwd_common(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* o, float* lse,
               const int32_t* cu, int nseq, int S, long long rows, int batch_dim, int Hq, int Hkv, int D, float scale,
               int window, void* stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    attn::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const int map_rows = (int)(cu ? rows : S);
    if (!make_map(&L.tq, q, D, Hq, map_rows, batch_dim) || !make_map(&L.tk, k, D, Hkv, map_rows, batch_dim) ||
        !make_map(&L.tv, v, D, Hkv, map_rows, batch_dim))
        return ATTN_ERR_LAUNCH;
    if (D == 512 && (Hq / Hkv) % 2 == 0) {
        if (!make_map(&L.tk_half, k, D, Hkv, map_rows, batch_dim, 64)) return ATTN_ERR_LAUNCH;
        L.pair_ok = true;
    }
    L.o = o, L.lse = lse, L.cu_seqlens = cu, L.status = dev->status;
    L.nseq = nseq, L.Hq = Hq, L.Hkv = Hkv, L.S = S, L.D = D, L.total_rows = (int)rows, L.window = window;
    L.scale = scale;
    return attn::launch_fwd(L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

// ---- launch accounting and the optional event profiler ------------------------------------
std::atomic<unsigned long long> g_launches{0};
std::mutex g_prof_mu;
bool g_prof_on = false;
struct ProfRec {
    const char* name;
    cudaEvent_t start, stop;
};
std::vector<ProfRec> g_prof;

}  // namespace

namespace attn {

ProfMark prof_begin(cudaStream_t stream, const char* kernel) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    ProfMark m;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (!g_prof_on) return m;
    ProfRec r{kernel, nullptr, nullptr};
    if (cudaEventCreate(&r.start) != cudaSuccess) return m;
    if (cudaEventCreate(&r.stop) != cudaSuccess) {
        cudaEventDestroy(r.start);
        return m;
    }
    cudaEventRecord(r.start, stream);
    m.slot = (int)g_prof.size();
    g_prof.push_back(r);
    return m;
}

void prof_end(cudaStream_t stream, ProfMark m) {
    if (m.slot < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (m.slot < (int)g_prof.size()) cudaEventRecord(g_prof[m.slot].stop, stream);
}

}  // namespace attn

namespace {
void prof_clear_locked() {
    for (auto& r : g_prof) {
        cudaEventDestroy(r.start);
        cudaEventDestroy(r.stop);
    }
    g_prof.clear();
}
}  // namespace

extern "C" {

unsigned long long attn_launch_count(void) { return g_launches.load(); }

int attn_profile_start(void) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof_clear_locked();
    g_prof_on = true;
    return ATTN_OK;
}

int attn_profile_stop(char* buf, size_t buf_bytes) {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof_on = false;
    struct Acc {
        long long n = 0;
        double ms = 0.0;
    };
    std::map<std::string, Acc> acc;
    int rc = 0;
    for (auto& r : g_prof) {
        float ms = 0.f;
        if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) {
            rc = -ATTN_ERR_LAUNCH;
            continue;
        }
        Acc& a = acc[r.name];
        a.n += 1;
        a.ms += ms;
    }
    prof_clear_locked();
    std::string out;
    for (auto& kv : acc) {
        char line[160];
        std::snprintf(line, sizeof(line), "%s %lld %.6f\n", kv.first.c_str(), kv.second.n, kv.second.ms);
        out += line;
    }
    if (buf && buf_bytes) {
        const size_t n = out.size() < buf_bytes - 1 ? out.size() : buf_bytes - 1;
        std::memcpy(buf, out.data(), n);
        buf[n] = 0;
    }
    return rc ? rc : (int)acc.size();
}


int attn_version(void) { return 100; }

const char* attn_status_string(int s) {
    switch (s) {
        case ATTN_OK: return "ATTN_OK";
        case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
        case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
        case ATTN_ERR_MISALIGNED: return "ATTN_ERR_MISALIGNED";
        case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
        case ATTN_ERR_LAUNCH: return "ATTN_ERR_LAUNCH";
        case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
        case ATTN_ERR_DEVICE_BOUNDS: return "ATTN_ERR_DEVICE_BOUNDS";
        case ATTN_ERR_NO_DEVICE: return "ATTN_ERR_NO_DEVICE";
        default: return "ATTN_ERR_UNKNOWN";
    }
}

size_t attn_workspace_size(int op, int B, int Hq, int Hkv, int S, int D, int num_seqs, int max_pages_per_seq) {
    (void)Hkv, (void)num_seqs, (void)max_pages_per_seq;
    if (B < 0 || Hq < 0 || S < 0 || D < 0) return 0;
    switch (op) {
        case ATTN_OP_FWD:
        case ATTN_OP_FWD_VARLEN: return 0;
        case ATTN_OP_BWD:
        case ATTN_OP_BWD_VARLEN: return bwd_ws((long long)B * S, Hq, D);
        case ATTN_OP_DECODE_PAGED: return decode_ws(B, Hq, Hkv, D);
        default: return 0;
    }
}

int attn_fwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* o, float* lse, int B, int Hq,
             int Hkv, int S, int D, float scale, int causal, int window, void* workspace, size_t workspace_bytes,
             void* stream) {
    (void)workspace, (void)workspace_bytes;
    if (!q || !k || !v || !o || !lse || B < 0 || S < 0) return ATTN_ERR_INVALID_ARG;
    int st = check_common(Hq, Hkv, scale, causal, window);
    if (st) return st;
    const long long rows = (long long)B * S;
    if ((st = check_prefill_shape(rows, Hq, Hkv, D, S))) return st;
    if (B > 65535 / fwd_splits(D)) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
    if (rows == 0) return ATTN_OK;
    return fwd_common(q, k, v, o, lse, nullptr, B, S, rows, B, Hq, Hkv, D, scale, window, stream);
}

int attn_fwd_varlen(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, attn_bf16* o, float* lse,
                    const int32_t* cu_seqlens, int num_seqs, int total_tokens, int max_seqlen, int Hq, int Hkv, int D,
                    float scale, int causal, int window, void* workspace, size_t workspace_bytes, void* stream) {
    (void)workspace, (void)workspace_bytes;
    if (!q || !k || !v || !o || !lse || !cu_seqlens || num_seqs < 0 || total_tokens < 0 || max_seqlen < 0)
        return ATTN_ERR_INVALID_ARG;
    int st = check_common(Hq, Hkv, scale, causal, window);
    if (st) return st;
    if ((st = check_prefill_shape(total_tokens, Hq, Hkv, D, max_seqlen))) return st;
    if (num_seqs > 65535 / fwd_splits(D)) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse)) return ATTN_ERR_MISALIGNED;
    if (num_seqs == 0 || total_tokens == 0 || max_seqlen == 0) return ATTN_OK;
    return fwd_common(q, k, v, o, lse, cu_seqlens, num_seqs, max_seqlen, total_tokens, 1, Hq, Hkv, D, scale, window,
                      stream);
}

int attn_fwd_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache, const int32_t* block_table,
                   const int32_t* seq_lens, const int32_t* cu_q, attn_bf16* o, float* lse, int num_reqs, int total_q,
                   int max_q_len, int Hq, int Hkv, int D, int page_size, int max_pages_per_seq, int num_pages,
                   float scale, int causal, int window, void* stream) {
    if (num_reqs < 0 || total_q < 0 || max_q_len < 0 || max_pages_per_seq < 0 || num_pages < 0 || page_size <= 0)
        return ATTN_ERR_INVALID_ARG;
    int st = check_common(Hq, Hkv, scale, causal, window);
    if (st) return st;
    if ((st = check_prefill_shape(total_q, Hq, Hkv, D, max_q_len))) return st;
    if (page_size != 16 || num_reqs > 65535 / fwd_splits(D) || max_pages_per_seq > (1 << 24)) return ATTN_ERR_UNSUPPORTED;
    if (num_reqs == 0 || total_q == 0 || max_q_len == 0) return ATTN_OK;  // nothing to read or write
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !cu_q || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
        (reinterpret_cast<uintptr_t>(cu_q) & 3u))
        return ATTN_ERR_MISALIGNED;
    if (num_pages == 0 || max_pages_per_seq == 0) return ATTN_ERR_INVALID_ARG;  // new tokens need cached pages
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    attn::FwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    if (!make_map(&L.tq, q, D, Hq, total_q, 1) || !make_cache_map(&L.tk, k_cache, D, Hkv, num_pages) ||
        !make_cache_map(&L.tv, v_cache, D, Hkv, num_pages))
        return ATTN_ERR_LAUNCH;
    if (D == 512) {  // CTA pairs: each CTA loads 4 pages x 256 columns of a key tile
        if (!make_cache_map(&L.tk_half, k_cache, D, Hkv, num_pages, 4)) return ATTN_ERR_LAUNCH;
        L.pair_ok = true;
    }
    L.o = o, L.lse = lse, L.cu_seqlens = nullptr, L.status = dev->status;
    L.nseq = num_reqs, L.Hq = Hq, L.Hkv = Hkv, L.S = max_q_len, L.D = D, L.total_rows = total_q, L.window = window;
    L.scale = scale;
    L.block_table = block_table, L.seq_lens = seq_lens, L.cu_q = cu_q;
    L.max_pages = max_pages_per_seq, L.num_pages = num_pages;
    return attn::launch_fwd(L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_bwd(const attn_bf16* q, const attn_bf16* k, const attn_bf16* v, const attn_bf16* o, const float* lse,
             const attn_bf16* dO, attn_bf16* dQ, attn_bf16* dK, attn_bf16* dV, int B, int Hq, int Hkv, int S, int D,
             float scale, int causal, int window, const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
             void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k || !v || !o || !lse || !dO || !dQ || !dK || !dV || B < 0 || S < 0) return ATTN_ERR_INVALID_ARG;
    int st = check_common(Hq, Hkv, scale, causal, window);
    if (st) return st;
    const bool varlen = cu_seqlens != nullptr;
    if (varlen && (B != 1 || num_seqs < 0 || max_seqlen < 0)) return ATTN_ERR_INVALID_ARG;
    const long long rows = (long long)B * S;
    const int grid_len = varlen ? max_seqlen : S;
    if ((st = check_prefill_shape(rows, Hq, Hkv, D, grid_len))) return st;
    if ((varlen ? num_seqs : B) > 65535) return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse) || !aligned16(dO) ||
        !aligned16(dQ) || !aligned16(dK) || !aligned16(dV))
        return ATTN_ERR_MISALIGNED;
    const size_t need = bwd_ws(rows, Hq, D);
    if (rows > 0 && (!workspace || workspace_bytes < need)) return ATTN_ERR_WORKSPACE;
    if (workspace && (reinterpret_cast<uintptr_t>(workspace) & 255u)) return ATTN_ERR_MISALIGNED;
    if (rows == 0 || (varlen && (num_seqs == 0 || max_seqlen == 0))) return ATTN_OK;
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    attn::BwdLaunch L;
    std::memset(&L, 0, sizeof(L));
    const int map_rows = varlen ? (int)rows : S, batch = varlen ? 1 : B;
    if (!make_map(&L.tq, q, D, Hq, map_rows, batch) || !make_map(&L.tk, k, D, Hkv, map_rows, batch) ||
        !make_map(&L.tv, v, D, Hkv, map_rows, batch) || !make_map(&L.tdo, dO, D, Hq, map_rows, batch))
        return ATTN_ERR_LAUNCH;
    // query-share maps of the cluster kernel (D >= 256 only)
    if (D >= 256 && (!make_map(&L.tqh, q, D, Hq, map_rows, batch, 256 * 128 / D) ||
                     !make_map(&L.tdoh, dO, D, Hq, map_rows, batch, 256 * 128 / D)))
        return ATTN_ERR_LAUNCH;
    L.q = q, L.k = k, L.v = v, L.o = o, L.dO = dO, L.lse = lse, L.dQ = dQ, L.dK = dK, L.dV = dV;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    L.dq_acc = reinterpret_cast<float*>(ws);
    if (!make_map_f32(&L.tdq, L.dq_acc, D, Hq, map_rows, batch)) return ATTN_ERR_LAUNCH;
    L.delta = reinterpret_cast<float*>(ws + align256((size_t)rows * Hq * D * 4));
    L.cu_seqlens = cu_seqlens, L.status = dev->status;
    L.nseq = varlen ? num_seqs : B;
    L.Hq = Hq, L.Hkv = Hkv, L.S = grid_len, L.D = D, L.total_rows = (int)rows, L.window = window, L.scale = scale;
    return attn::launch_bwd(L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_decode_paged(const attn_bf16* q, const attn_bf16* k_cache, const attn_bf16* v_cache,
                      const int32_t* block_table, const int32_t* seq_lens, attn_bf16* o, float* lse, int B, int Hq,
                      int Hkv, int D, int page_size, int max_pages_per_seq, int num_pages, float scale, int window,
                      void* workspace, size_t workspace_bytes, void* stream) {
    if (!q || !k_cache || !v_cache || !block_table || !seq_lens || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (B < 0 || max_pages_per_seq < 0 || num_pages < 0 || page_size <= 0 || window < 0) return ATTN_ERR_INVALID_ARG;
    if (Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0) return ATTN_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
    const int G = Hq / Hkv;
    if (!decode_shape_ok(Hq, Hkv, D) || page_size != 16 || Hkv > 256 || B > 4096 || num_pages > (1 << 26))
        return ATTN_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) || !aligned16(lse) ||
        (reinterpret_cast<uintptr_t>(block_table) & 3u) || (reinterpret_cast<uintptr_t>(seq_lens) & 3u))
        return ATTN_ERR_MISALIGNED;
    if (B == 0) return ATTN_OK;
    if (!workspace || workspace_bytes < decode_ws(B, Hq, Hkv, D)) return ATTN_ERR_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255u) return ATTN_ERR_MISALIGNED;
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    attn::DecodeLaunch L;
    std::memset(&L, 0, sizeof(L));
    const int hb = attn::decode_heads_per_unit(Hkv, D, G), nhb = Hkv / hb;
    if (attn::decode_packed_layout(G, D)) {
        if (!make_decode_swz_map(&L.tk, k_cache, D, Hkv, num_pages, hb) ||
            !make_decode_swz_map(&L.tv, v_cache, D, Hkv, num_pages, hb))
            return ATTN_ERR_LAUNCH;
    } else if (nhb > 1 && (!make_decode_map(&L.tk, k_cache, D, Hkv, num_pages, hb) ||
                           !make_decode_map(&L.tv, v_cache, D, Hkv, num_pages, hb))) {
        return ATTN_ERR_LAUNCH;
    }
    L.q = q, L.k_cache = k_cache, L.v_cache = v_cache, L.block_table = block_table, L.seq_lens = seq_lens;
    L.o = o, L.lse = lse, L.status = dev->status;
    uint8_t* ws = static_cast<uint8_t*>(workspace);
    L.part = reinterpret_cast<float*>(ws);
    L.B = B, L.Hq = Hq, L.Hkv = Hkv, L.D = D, L.max_pages = max_pages_per_seq, L.num_pages = num_pages;
    L.scale = scale, L.window = window;
    // the head blocks share the SMs: each block's pages are split over sms / nhb CTAs
    long long units = (long long)B * (max_pages_per_seq > 0 ? max_pages_per_seq : 1);
    int grid = dev->sms / nhb;
    if (grid > decode_grid_cap(nhb)) grid = decode_grid_cap(nhb);
    if (units < grid) grid = (int)units;
    L.grid = grid < 1 ? 1 : grid;
    return attn::launch_decode_paged(L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_merge_lse(const attn_bf16* o_parts, const float* lse_parts, attn_bf16* o, float* lse, int num_parts, int B,
                   int S, int H, int D, void* stream) {
    if (num_parts < 1 || B < 0 || S < 0 || H < 1) return ATTN_ERR_INVALID_ARG;
    if ((D != 64 && D != 128 && D != 256 && D != 512) || num_parts > 64) return ATTN_ERR_UNSUPPORTED;
    const long long rows = (long long)B * S * H;
    if (rows == 0) return ATTN_OK;
    if (!o_parts || !lse_parts || !o || !lse) return ATTN_ERR_INVALID_ARG;
    if (!aligned16(o_parts) || !aligned16(o) || (reinterpret_cast<uintptr_t>(lse_parts) & 3u) ||
        (reinterpret_cast<uintptr_t>(lse) & 3u))
        return ATTN_ERR_MISALIGNED;
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    attn::MergeLaunch L;
    L.o_parts = o_parts, L.lse_parts = lse_parts, L.o = o, L.lse = lse;
    L.P = num_parts, L.B = B, L.S = S, L.H = H, L.D = D, L.sms = dev->sms;
    return attn::launch_merge_lse(L, static_cast<cudaStream_t>(stream)) == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_selftest_wait_timeout(int limit_ms, void* stream) {
    if (limit_ms < 1 || limit_ms > 10000) return ATTN_ERR_INVALID_ARG;
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    const attn::ProfMark m = attn::prof_begin(static_cast<cudaStream_t>(stream), "selftest_wait");
    selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->status,
                                                                          (unsigned long long)limit_ms * 1000000ull);
    attn::prof_end(static_cast<cudaStream_t>(stream), m);
    return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_LAUNCH;
}

int attn_get_device_status(void* stream) {
    const DeviceInfo* dev = device_info();
    if (!dev) return ATTN_ERR_NO_DEVICE;
    if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return ATTN_ERR_LAUNCH;
    unsigned words[2] = {0u, 0u}, zero[2] = {0u, 0u};
    if (cudaMemcpyFromSymbol(words, g_attn_status, sizeof(words)) != cudaSuccess) return ATTN_ERR_LAUNCH;
    if ((words[0] || words[1]) && cudaMemcpyToSymbol(g_attn_status, zero, sizeof(zero)) != cudaSuccess)
        return ATTN_ERR_LAUNCH;
    const unsigned flags = words[0];
    if (flags && std::getenv("ATTN_DEBUG"))
        std::fprintf(stderr, "attn: device status flags=0x%x first timed-out wait site=0x%x\n", flags, words[1]);
    if (flags & attn::DEVSTAT_TIMEOUT) return ATTN_ERR_DEVICE_TIMEOUT;
    if (flags & attn::DEVSTAT_BOUNDS) return ATTN_ERR_DEVICE_BOUNDS;
    return ATTN_OK;
}

}  // extern "C"
