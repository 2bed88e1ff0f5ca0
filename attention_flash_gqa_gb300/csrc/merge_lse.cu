// Merge of attention results over disjoint key sets: the combining step of context-parallel
// ring attention.
//
// Source: "Gemma4 FFPA attention backend support ...", "Integration": under context
// parallelism every ring chunk of keys is attended separately by the fused kernel (dense or
// varlen per chunk), and the chunks' results make up the attention over all keys. Each part p
// holds o_p, normalised over its own keys, and lse_p, the natural log of the sum of exp(score)
// over those keys. The attention over the union of the keys is
//     lse = ln sum_p exp(lse_p),   o = sum_p exp(lse_p - lse) o_p
// evaluated with the largest lse_p factored out. A part with lse_p = -inf had no allowed key
// and contributes nothing (its o_p is never multiplied in, even if it holds NaN). A row where
// every part is empty gets o = 0 and lse = -inf.
//
// Memory bound: every byte of every part is read once. D/8 threads share a row, each owning one
// 16-byte vector (8 dims) of it, so a 256-thread block covers 256 / (D/8) rows per pass. Rows
// are walked in the lse layout's order (b, h, s), so the lse loads of a pass are coalesced; each
// row of o is contiguous. The threads of a row walk the parts kChunk at a time: the chunk's lse
// values (broadcast loads) and 16-byte vectors are all in flight before any is used, and the
// running maximum, weight sum and fp32 accumulator are rescaled once per chunk. Two parts per
// chunk measured fastest (5.1 TB/s for 8 parts of 2048 x 32 x 512, against 4.4 with eight):
// the smaller register footprint keeps more threads, and so more loads, resident per SM.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cmath>

#include "attn_internal.h"

namespace attn {
namespace {

constexpr int kThreads = 256;
constexpr int kChunk = 2;  // parts whose loads are in flight together (more resident threads beat deeper chunks)

struct MergeArgs {
    const uint16_t* o_parts;  // [P, B, S, H, D]
    const float* lse_parts;   // [P, B, H, S]
    uint16_t* o;              // [B, S, H, D]
    float* lse;               // [B, H, S]
    long long rows;           // B * H * S
    int P, S, H, D;
};

__device__ __forceinline__ float lo_bf16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi_bf16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }
__device__ __forceinline__ uint32_t pack2(float a, float b) {
    const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&v);
}

template <int TPR>  // threads per row = D / 8
__global__ void __launch_bounds__(kThreads) merge_lse_kernel(MergeArgs a) {
    constexpr int RPB = kThreads / TPR;  // rows per pass
    const int rsub = threadIdx.x / TPR, vec = threadIdx.x % TPR;
    const long long passes = (a.rows + RPB - 1) / RPB;
    const size_t part_o = (size_t)a.rows * a.D;
    const size_t part_l = (size_t)a.rows;
    for (long long pass = blockIdx.x; pass < passes; pass += gridDim.x) {  // uniform over the block
        const long long r = pass * RPB + rsub;  // row in (b, h, s) order = its lse index
        const bool valid = r < a.rows;
        // running merge over the parts, kChunk at a time: m = largest lse so far, sum =
        // sum exp(lse_p - m), acc = sum exp(lse_p - m) o_p; at the end lse = m + ln sum and
        // o = acc / sum (the same weights exp(lse_p - lse), factored differently)
        float m = -INFINITY, sum = 0.f;
        float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        size_t orow = 0;
        if (valid) {
            const long long bh = r / a.S;
            const int s = (int)(r - bh * a.S);
            const int h = (int)(bh % a.H);
            const long long b = bh / a.H;
            orow = ((size_t)(b * a.S + s) * a.H + h) * a.D + (size_t)vec * 8;
            for (int p0 = 0; p0 < a.P; p0 += kChunk) {
                // every load of the chunk is issued before any of them is used
                float x[kChunk];
                uint4 w[kChunk];
#pragma unroll
                for (int u = 0; u < kChunk; ++u) {
                    const bool in = p0 + u < a.P;
                    x[u] = in ? a.lse_parts[(p0 + u) * part_l + r] : -INFINITY;
                    w[u] = in ? *reinterpret_cast<const uint4*>(a.o_parts + (p0 + u) * part_o + orow)
                              : make_uint4(0u, 0u, 0u, 0u);
                }
                float cm = m;
#pragma unroll
                for (int u = 0; u < kChunk; ++u) cm = fmaxf(cm, x[u]);
                if (cm == -INFINITY) continue;  // no key in any part so far
                const float rescale = m == -INFINITY ? 0.f : expf(m - cm);
                sum *= rescale;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc[e] *= rescale;
#pragma unroll
                for (int u = 0; u < kChunk; ++u) {
                    if (x[u] > -INFINITY) {  // an empty part's o is never multiplied in
                        const float wt = expf(x[u] - cm);
                        sum += wt;
                        const uint32_t ws[4] = {w[u].x, w[u].y, w[u].z, w[u].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc[2 * e] = fmaf(wt, lo_bf16(ws[e]), acc[2 * e]);
                            acc[2 * e + 1] = fmaf(wt, hi_bf16(ws[e]), acc[2 * e + 1]);
                        }
                    }
                }
                m = cm;
            }
        }
        const float L = m == -INFINITY ? -INFINITY : m + logf(sum);
        const float inv = m == -INFINITY ? 0.f : 1.f / sum;
        // Every read of this pass precedes its writes, so o / lse may be part 0's own buffers
        // (an in-place running merge): each o vector is read and written by one thread, and a
        // row's lse parts are read by all of its threads before one of them writes lse.
        __syncthreads();
        if (valid) {
            uint4 out;
            out.x = pack2(acc[0] * inv, acc[1] * inv);
            out.y = pack2(acc[2] * inv, acc[3] * inv);
            out.z = pack2(acc[4] * inv, acc[5] * inv);
            out.w = pack2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4*>(a.o + orow) = out;
            if (vec == 0) a.lse[r] = L;
        }
    }
}

template <int TPR>
cudaError_t launch_t(const MergeArgs& a, long long passes, int sms, cudaStream_t stream) {
    int per_sm = 0;  // resident blocks per SM (registers bound it): one wave of the grid-stride loop
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, merge_lse_kernel<TPR>, kThreads, 0);
    if (e != cudaSuccess) return e;
    const long long cap = (long long)sms * (per_sm > 0 ? per_sm : 1);
    const int grid = (int)(passes < cap ? passes : cap);
    const ProfMark m = prof_begin(stream, "merge_lse");
    merge_lse_kernel<TPR><<<grid, kThreads, 0, stream>>>(a);
    prof_end(stream, m);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_merge_lse(const MergeLaunch& L, cudaStream_t stream) {
    MergeArgs a;
    a.o_parts = L.o_parts, a.lse_parts = L.lse_parts, a.o = L.o, a.lse = L.lse;
    a.rows = (long long)L.B * L.H * L.S;
    a.P = L.P, a.S = L.S, a.H = L.H, a.D = L.D;
    if (a.rows == 0) return cudaSuccess;
    const int tpr = L.D / 8;
    const long long passes = (a.rows + (kThreads / tpr) - 1) / (kThreads / tpr);
    switch (tpr) {
        case 8: return launch_t<8>(a, passes, L.sms, stream);
        case 16: return launch_t<16>(a, passes, L.sms, stream);
        case 32: return launch_t<32>(a, passes, L.sms, stream);
        case 64: return launch_t<64>(a, passes, L.sms, stream);
        default: return cudaErrorInvalidValue;
    }
}

}  // namespace attn
