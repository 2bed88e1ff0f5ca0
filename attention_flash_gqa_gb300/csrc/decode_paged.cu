// Single-token decode over a paged KV cache (D = 128, page = 16 tokens).
//
// Source: "flex_attention + paged KV + CUDA graphs vs vLLM", sections "What each
// option did" (page-table indirection per block, contiguous blocks, more warps) and
// "Architecture notes" (PagedKVCache + PageTable); "What broke correctness" (a row
// whose mask has no allowed key must not produce NaN).
//
// Design (memory bound: every cached K/V byte is read exactly once):
//  * A page holds 16 tokens x Hkv heads x 128 dims, contiguous, so one page of K and
//    one of V are fetched with two untiled TMA bulk copies into a 3-stage ring.
//  * Work is balanced by pages, not by requests: the pages of all requests are laid
//    end to end and CTA k takes the k-th equal share. A CTA may cover the tail of one
//    request and the head of the next.
//  * 16 consumer warps, two per KV head: each serves all query heads of the head's GQA
//    group (one K/V row read feeds all of them) on one half of the page's 16 tokens, with
//    its own running softmax state. Lane l owns dims 4l..4l+3; per-token dot products are
//    finished by a butterfly reduce-scatter across the warp.
//  * fp32 online softmax in the log2 domain. Every (CTA, token half) touching a request
//    leaves unnormalised partials (o, m, l) in the workspace; the last CTA to finish that
//    request (arrival counter) merges them and resets the counter to zero.
#include <cuda_runtime.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kD = 128;
constexpr int kPage = 16;
constexpr int kStages = 3;
constexpr int kConsumerWarps = 16;
constexpr int kThreads = (kConsumerWarps + 1) * 32;  // + one producer warp
constexpr int kMaxB = 4096;
constexpr int kRowF = kD + 4;
constexpr int kMaxUnits = 2048;  // page-table entries of a CTA's range staged in shared memory  // partial row: o[kD], m, l, 2 pad floats (keeps float4 alignment)

struct DecodeArgs {
    const uint16_t* q;
    const uint16_t* kc;
    const uint16_t* vc;
    const int32_t* block_table;
    const int32_t* seq_lens;
    uint16_t* o;
    float* lse;
    float* part;       // [(B + grid) * 2 slots][Hq][kRowF]
    int32_t* counters; // [B]
    unsigned* status;
    int B, Hq, Hkv, max_pages, num_pages;
    float scale_log2;
};

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Clamped page count of request b (records a bounds fault for lengths beyond the table).
__device__ __forceinline__ int req_len(const DecodeArgs& a, int b) {
    int L = a.seq_lens[b];
    int cap = a.max_pages * kPage;
    if (L < 0 || L > cap) {
        atomicOr(a.status, DEVSTAT_BOUNDS);
        L = L < 0 ? 0 : cap;
    }
    return L;
}

// CTA that owns global page unit u when P units are split evenly over G CTAs
// (CTA k owns [floor(kP/G), floor((k+1)P/G))).
__device__ __forceinline__ int owner_of(long long u, long long P, int G) {
    return (int)(((u + 1) * (long long)G - 1) / P);
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) decode_paged_kernel(DecodeArgs a) {
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const int page_bytes = kPage * a.Hkv * kD * 2;
    uint8_t* stage_base = smem;  // kStages x (K page, V page)
    int32_t* start = reinterpret_cast<int32_t*>(smem + kStages * 2 * page_bytes);  // [B + 1]
    float* scratch = reinterpret_cast<float*>(start + kMaxB + 8);                  // per warp: sc[8G], sp[8G]
    uint64_t* bars = reinterpret_cast<uint64_t*>(scratch + kConsumerWarps * 16 * 8);
    uint64_t* full = bars;
    uint64_t* empty = bars + kStages;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 2 * kStages);
    int* last_flag = const_cast<int*>(abort_flag) + 1;
    int* warp_sums = last_flag + 1;  // [8]
    int32_t* unit_tab = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(bars) + 256);  // [kMaxUnits]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = a.B;

    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }

    // ---- page prefix sums over requests: start[b] = pages before request b ----------
    {
        const int per = (B + 255) / 256;
        int local = 0;
        if (tid < 256) {
            for (int i = 0; i < per; ++i) {
                int b = tid * per + i;
                if (b < B) local += (req_len(a, b) + kPage - 1) / kPage;
            }
        }
        // inclusive scan of `local` over threads 0..255
        int v = local;
        for (int off = 1; off < 32; off <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, v, off);
            if (lane >= off) v += n;
        }
        if (tid < 256 && lane == 31) warp_sums[warp] = v;
        __syncthreads();
        int before = 0;
        if (tid < 256)
            for (int w = 0; w < warp; ++w) before += warp_sums[w];
        int excl = before + v - local;
        if (tid < 256) {
            int acc = excl;
            for (int i = 0; i < per; ++i) {
                int b = tid * per + i;
                if (b < B) {
                    start[b] = acc;
                    acc += (req_len(a, b) + kPage - 1) / kPage;
                }
            }
            if (tid == 255) start[B] = acc;
        }
        __syncthreads();
    }
    const long long P = start[B];
    // Pages are shared by Gc = min(grid, P) CTAs, so every participating CTA owns at
    // least one page and the CTAs touching a request are exactly owner(first)..owner(last).
    const int Gc = (int)(P < (long long)gridDim.x ? P : (long long)gridDim.x);
    const int k = blockIdx.x;

    // Requests with no cached token: o = 0, lse = -inf (CTA 0 writes them).
    if (k == 0) {
        for (int idx = tid; idx < B * a.Hq; idx += kThreads) {
            int b = idx / a.Hq;
            if (start[b + 1] == start[b]) {
                a.lse[idx] = -INFINITY;
                uint16_t* orow = a.o + (size_t)idx * kD;
                for (int d = 0; d < kD; d += 8) *reinterpret_cast<uint4*>(orow + d) = make_uint4(0, 0, 0, 0);
            }
        }
    }
    if (P == 0 || k >= Gc) return;
    const long long u0 = (long long)k * P / Gc, u1 = (long long)(k + 1) * P / Gc;
    if (u0 >= u1) return;

    // first request overlapping [u0, u1): largest b with start[b] <= u0 and a nonempty range
    int b_first = 0;
    {
        int lo = 0, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= u0) lo = mid;
            else hi = mid - 1;
        }
        b_first = lo;
        while (b_first < B && start[b_first + 1] <= u0) ++b_first;
    }

    // Page table of this CTA's range, gathered once by all threads: entry = page id << 5 |
    // valid tokens in the page (1..16), or -1 for a page id outside the pool. The loops below
    // then never wait on a dependent global load.
    const int n_units = (int)(u1 - u0);
    auto make_entry = [&](int kk) -> int32_t {
        const long long u = u0 + kk;
        int lo = b_first, hi = B - 1;
        while (lo < hi) {
            int mid = (lo + hi + 1) >> 1;
            if (start[mid] <= u) lo = mid;
            else hi = mid - 1;
        }
        const int p = (int)(u - start[lo]);
        const int page = a.block_table[(size_t)lo * a.max_pages + p];
        if (page < 0 || page >= a.num_pages) {
            atomicOr(a.status, DEVSTAT_BOUNDS);
            return -1;
        }
        const int nt = min(kPage, req_len(a, lo) - p * kPage);
        return (page << 5) | nt;
    };
    for (int kk = tid; kk < n_units && kk < kMaxUnits; kk += kThreads) unit_tab[kk] = make_entry(kk);
    __syncthreads();
    auto unit_entry = [&](int kk) -> int32_t { return kk < kMaxUnits ? unit_tab[kk] : make_entry(kk); };

    if (warp == kConsumerWarps) {
        // ---------------------------- producer ------------------------------------------
        if (lane == 0) {
            int b = b_first;
            int i = 0;
            for (long long u = u0; u < u1; ++u, ++i) {
                while (start[b + 1] <= u) ++b;
                const int s = i % kStages, r = i / kStages;
                if (r > 0 && !mbar_wait(smem_u32(&empty[s]), (r - 1) & 1, abort_flag, a.status, 0x31)) break;
                const int32_t entry = unit_entry(i);
                const uint32_t fb = smem_u32(&full[s]);
                if (entry >= 0) {
                    mbar_expect_tx(fb, 2u * page_bytes);
                    const size_t off = (size_t)(entry >> 5) * kPage * a.Hkv * kD;
                    bulk_load(smem_u32(stage_base + (size_t)s * 2 * page_bytes), a.kc + off, page_bytes, fb);
                    bulk_load(smem_u32(stage_base + (size_t)s * 2 * page_bytes + page_bytes), a.vc + off, page_bytes, fb);
                } else {
                    mbar_arrive(fb);
                }
            }
            // Drain: every issued copy completes before this CTA may exit.
            const int issued = i;
            for (int s = 0; s < kStages && s < issued; ++s) {
                const int last = s + ((issued - 1 - s) / kStages) * kStages;
                mbar_drain(smem_u32(&full[s]), (last / kStages) & 1, a.status, 0x33);
            }
        }
        return;
    }

    // ---------------------------------- consumers ----------------------------------------
    // Warp w serves KV head w / 2 for all G query heads of its group, on tokens
    // 8 * (w % 2) .. 8 * (w % 2) + 7 of every page: the two warps of a head keep separate
    // running softmax states and are merged like split partials at the end.
    const int g = warp >> 1, half = warp & 1;
    const bool active = g < a.Hkv;
    float* sc = scratch + warp * 16 * G;  // [8 * G] scores (log2 domain)
    float* sp = sc + 8 * G;               // [8 * G] probabilities
    constexpr int NV = 8 * G;             // (token, head) values per half page
    constexpr int NF = NV >= 32 ? NV / 32 : 1;
    constexpr int KH = NV >= 32 ? 5 : (NV == 16 ? 4 : (NV == 8 ? 3 : 2));  // halving steps
    constexpr int NH = NV >= 32 ? NV / 32 : 1;  // values per lane in the softmax layout

    // Query rows: lane holds dims 4*lane .. 4*lane+3 of each of the G heads.
    float qv[G][4];  // loaded when the request changes
    for (int hh = 0; hh < G; ++hh)
        for (int e = 0; e < 4; ++e) qv[hh][e] = 0.f;
    float m_run = -INFINITY, l_run = 0.f;  // for head (lane % G)
    float acc_o[G][4];
    for (int hh = 0; hh < G; ++hh)
        for (int e = 0; e < 4; ++e) acc_o[hh][e] = 0.f;

    int b = b_first;
    int i = 0;
    bool ok = true;
    int cur_b = -1;
    for (long long u = u0; u < u1 && ok; ++u, ++i) {
        while (start[b + 1] <= u) ++b;
        if (b != cur_b) {
            cur_b = b;
            if (active) {
                for (int hh = 0; hh < G; ++hh) {
                    const uint2 w = *reinterpret_cast<const uint2*>(a.q + ((size_t)b * a.Hq + g * G + hh) * kD + 4 * lane);
                    qv[hh][0] = bf16_lo(w.x), qv[hh][1] = bf16_hi(w.x), qv[hh][2] = bf16_lo(w.y), qv[hh][3] = bf16_hi(w.y);
                }
            }
        }
        const int s = i % kStages, r = i / kStages;
        ok = mbar_wait(smem_u32(&full[s]), r & 1, abort_flag, a.status, 0x32);
        if (!ok) break;
        const int32_t entry = unit_entry(i);
        const int nt = (entry >= 0 ? (entry & 31) : 0) - 8 * half;  // valid tokens of this half (may be <= 0)
        if (active && nt > 0) {
            const uint8_t* kp = stage_base + (size_t)s * 2 * page_bytes + (size_t)8 * half * a.Hkv * kD * 2;
            const uint8_t* vp = kp + page_bytes;
            // scores: v[t*G + hh], partial over this lane's 4 dims
            float v[NV];
#pragma unroll
            for (int t = 0; t < 8; ++t) {
                const uint2 w = *reinterpret_cast<const uint2*>(kp + ((size_t)(t * a.Hkv + g) * kD + 4 * lane) * 2);
                const float k0 = bf16_lo(w.x), k1 = bf16_hi(w.x), k2 = bf16_lo(w.y), k3 = bf16_hi(w.y);
#pragma unroll
                for (int hh = 0; hh < G; ++hh)
                    v[t * G + hh] = qv[hh][0] * k0 + qv[hh][1] * k1 + qv[hh][2] * k2 + qv[hh][3] * k3;
            }
            // butterfly reduce-scatter over lane offsets 16, 8, 4, 2, 1: after KH halvings a lane
            // holds NF values, index (lane >> (5 - KH)) * NF + j; remaining offsets all-reduce.
            int count = NV;
#pragma unroll
            for (int off = 16; off >= 1; off >>= 1) {
                if (count > 1) {
                    const int hf = count >> 1;
                    const bool upper = (lane & off) != 0;
#pragma unroll
                    for (int j = 0; j < NV / 2; ++j) {
                        if (j < hf) {
                            const float send = upper ? v[j] : v[hf + j];
                            const float keep = upper ? v[hf + j] : v[j];
                            v[j] = keep + __shfl_xor_sync(0xffffffffu, send, off);
                        }
                    }
                    count = hf;
                } else {
                    v[0] += __shfl_xor_sync(0xffffffffu, v[0], off);
                }
            }
            if ((lane & ((1 << (5 - KH)) - 1)) == 0) {
#pragma unroll
                for (int j = 0; j < NF; ++j) {
                    const int idx = (lane >> (5 - KH)) * NF + j;
                    sc[idx] = idx / G < nt ? v[j] * a.scale_log2 : -INFINITY;
                }
            }
            __syncwarp();
            // softmax layout: lane holds idx = lane + 32*j (head lane % G, token idx / G)
            float sv[NH];
            float mx = -INFINITY;
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                const int idx = lane + 32 * j;
                sv[j] = idx < NV ? sc[idx] : -INFINITY;
                mx = fmaxf(mx, sv[j]);
            }
#pragma unroll
            for (int off = G; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
            const float m_new = fmaxf(m_run, mx);
            const float m_use = m_new == -INFINITY ? 0.f : m_new;
            const float alpha = m_run == -INFINITY ? (m_new == -INFINITY ? 1.f : 0.f) : fast_exp2(m_run - m_use);
            float psum = 0.f;
#pragma unroll
            for (int j = 0; j < NH; ++j) {
                const int idx = lane + 32 * j;
                const float pj = sv[j] == -INFINITY ? 0.f : fast_exp2(sv[j] - m_use);
                if (idx < NV) sp[idx] = pj;
                psum += pj;
            }
#pragma unroll
            for (int off = G; off < 32; off <<= 1) psum += __shfl_xor_sync(0xffffffffu, psum, off);
            l_run = l_run * alpha + psum;
            m_run = m_new;
            __syncwarp();
            // o update: lane's 4 dims for all G heads
#pragma unroll
            for (int hh = 0; hh < G; ++hh) {
                const float al = __shfl_sync(0xffffffffu, alpha, hh);
#pragma unroll
                for (int e = 0; e < 4; ++e) acc_o[hh][e] *= al;
            }
            const int tmax = nt < 8 ? nt : 8;
            for (int t = 0; t < tmax; ++t) {
                const uint2 w = *reinterpret_cast<const uint2*>(vp + ((size_t)(t * a.Hkv + g) * kD + 4 * lane) * 2);
                const float v0 = bf16_lo(w.x), v1 = bf16_hi(w.x), v2 = bf16_lo(w.y), v3 = bf16_hi(w.y);
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    const float pt = sp[t * G + hh];
                    acc_o[hh][0] += pt * v0, acc_o[hh][1] += pt * v1, acc_o[hh][2] += pt * v2, acc_o[hh][3] += pt * v3;
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(&empty[s]));

        // ---- end of this request inside this CTA: write partials, last CTA merges -------
        const long long req_end = start[b + 1];
        if (u + 1 == req_end || u + 1 == u1) {
            const int kf = owner_of(start[b], P, Gc), kl = owner_of(req_end - 1, P, Gc);
            // slot of (request b, CTA k, token half): (b + k) * 2 + half
            float* slot = a.part + ((size_t)(b + k) * 2 + half) * a.Hq * kRowF;
            if (active) {
#pragma unroll
                for (int hh = 0; hh < G; ++hh) {
                    float* row = slot + (size_t)(g * G + hh) * kRowF;
                    *reinterpret_cast<float4*>(row + 4 * lane) =
                        make_float4(acc_o[hh][0], acc_o[hh][1], acc_o[hh][2], acc_o[hh][3]);
                    if (lane == hh) {
                        row[kD] = m_run;
                        row[kD + 1] = l_run;
                    }
                }
            }
            __threadfence();
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            if (tid == 0) {
                const int prev = atomicAdd(&a.counters[b], 1);
                *last_flag = prev == kl - kf;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            if (*last_flag) {
                __threadfence();
                // merge the partials of CTAs kf..kl (both token halves) for every (head, dim)
                const int nslots = 2 * (kl - kf + 1);
                for (int idx = tid; idx < a.Hq * (kD / 4); idx += kConsumerWarps * 32) {
                    const int h = idx / (kD / 4), d4 = idx % (kD / 4);
                    float M = -INFINITY;
                    for (int q = 0; q < nslots; ++q) {
                        const float* row = a.part + ((size_t)(b + kf) * 2 + q) * a.Hq * kRowF + (size_t)h * kRowF;
                        M = fmaxf(M, __ldcg(row + kD));
                    }
                    const float Mu = M == -INFINITY ? 0.f : M;
                    float Ls = 0.f;
                    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
                    for (int q = 0; q < nslots; ++q) {
                        const float* row = a.part + ((size_t)(b + kf) * 2 + q) * a.Hq * kRowF + (size_t)h * kRowF;
                        const float mk = __ldcg(row + kD);
                        const float wgt = mk == -INFINITY ? 0.f : fast_exp2(mk - Mu);
                        Ls += wgt * __ldcg(row + kD + 1);
                        const float4 ov = __ldcg(reinterpret_cast<const float4*>(row) + d4);
                        O.x += wgt * ov.x, O.y += wgt * ov.y, O.z += wgt * ov.z, O.w += wgt * ov.w;
                    }
                    const float inv = Ls > 0.f ? 1.f / Ls : 0.f;
                    uint2 w;
                    w.x = pack_bf16x2(O.x * inv, O.y * inv);
                    w.y = pack_bf16x2(O.z * inv, O.w * inv);
                    *reinterpret_cast<uint2*>(a.o + ((size_t)b * a.Hq + h) * kD + 4 * d4) = w;
                    if (d4 == 0)
                        a.lse[(size_t)b * a.Hq + h] = Ls > 0.f ? (M + __log2f(Ls)) * 0.69314718055994531f : -INFINITY;
                }
                if (tid == 0) a.counters[b] = 0;
            }
            asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
            // reset the running state for the next request
            m_run = -INFINITY, l_run = 0.f;
            for (int hh = 0; hh < G; ++hh)
                for (int e = 0; e < 4; ++e) acc_o[hh][e] = 0.f;
        }
    }
}

}  // namespace

size_t decode_smem_bytes(int Hkv) {
    return 1024 + (size_t)kStages * 2 * kPage * Hkv * kD * 2 + (kMaxB + 8) * 4 + (size_t)kConsumerWarps * 16 * 8 * 4 +
           256 + kMaxUnits * 4;
}

int decode_max_grid() { return 256; }
int decode_row_floats() { return kRowF; }

cudaError_t launch_decode_paged(const DecodeLaunch& L, cudaStream_t stream) {
    DecodeArgs a;
    a.q = L.q, a.kc = L.k_cache, a.vc = L.v_cache, a.block_table = L.block_table, a.seq_lens = L.seq_lens;
    a.o = L.o, a.lse = L.lse, a.part = L.part, a.counters = L.counters, a.status = L.status;
    a.B = L.B, a.Hq = L.Hq, a.Hkv = L.Hkv, a.max_pages = L.max_pages, a.num_pages = L.num_pages;
    a.scale_log2 = L.scale * 1.4426950408889634f;
    const int G = L.Hq / L.Hkv;
    const size_t smem = decode_smem_bytes(L.Hkv);
    auto go = [&](auto kern) -> cudaError_t {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        const ProfMark m = prof_begin(stream, "decode_paged");
        kern<<<L.grid, kThreads, smem, stream>>>(a);
        prof_end(stream, m);
        return cudaGetLastError();
    };
    switch (G) {
        case 1: return go(decode_paged_kernel<1>);
        case 2: return go(decode_paged_kernel<2>);
        case 4: return go(decode_paged_kernel<4>);
        case 8: return go(decode_paged_kernel<8>);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
