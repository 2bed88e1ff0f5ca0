// Internal launch interfaces between the host API (api.cu) and the kernel files.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace attn {

// ---- launch accounting (api.cu) ------------------------------------------------------------
// Every kernel launch of the library goes through these: a process-wide launch counter and,
// when profiling is on, a CUDA event pair on the launching stream.
struct ProfMark {
    int slot = -1;
};
ProfMark prof_begin(cudaStream_t stream, const char* kernel);
void prof_end(cudaStream_t stream, ProfMark m);

// ---- paged decode -----------------------------------------------------------------------
struct DecodeLaunch {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *block_table, *seq_lens;
    uint16_t* o;
    float* lse;
    float* part;
    int32_t* counters;
    unsigned* status;
    int B, Hq, Hkv, max_pages, num_pages, grid;
    float scale;
};
size_t decode_smem_bytes(int Hkv);
int decode_max_grid();
int decode_row_floats();  // floats per (slot, head) partial row
cudaError_t launch_decode_paged(const DecodeLaunch& L, cudaStream_t stream);

// ---- prefill forward ---------------------------------------------------------------------
// q/k/v tensor maps are 4-D over [D, H, S, B] (varlen: B = 1, S = total tokens) with a
// 64 x 1 x 128 x 1 box and 128-byte swizzle.
struct FwdLaunch {
    CUtensorMap tq, tk, tv;
    uint16_t* o;
    float* lse;
    const int32_t* cu_seqlens;  // null: dense
    unsigned* status;
    int nseq;                   // B (dense) or num_seqs (varlen)
    int Hq, Hkv, S, D;          // S: dense sequence length or max_seqlen (varlen)
    int total_rows;             // B*S (dense) or total tokens (varlen)
    int window;
    float scale;
};
cudaError_t launch_fwd(const FwdLaunch& L, cudaStream_t stream);

// ---- backward ---------------------------------------------------------------------------
struct BwdLaunch {
    CUtensorMap tq, tk, tv, tdo;
    CUtensorMap tqh, tdoh;  // q / dO with a 64 x 1 x (256*128/D) x 1 box: one cluster CTA's query share
    CUtensorMap tdq;  // fp32 dQ accumulator, 4-D [D, Hq, S, B], box 32 x 1 x 128 x 1, 128-byte swizzle
    const uint16_t *q, *k, *v, *o, *dO;
    const float* lse;
    uint16_t *dQ, *dK, *dV;
    float* dq_acc;  // [rows, Hq, D] fp32
    float* delta;   // same layout as lse
    const int32_t* cu_seqlens;
    unsigned* status;
    int nseq, Hq, Hkv, S, D, total_rows, window;
    float scale;
};
cudaError_t launch_bwd(const BwdLaunch& L, cudaStream_t stream);

}  // namespace attn
