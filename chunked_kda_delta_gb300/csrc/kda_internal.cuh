// kda_internal.cuh -- declarations shared by the library's translation units
// (host API and kernels).  Not part of the public ABI; see include/kda.h.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace kda {

constexpr int kD = 128;     // Dk = Dv
constexpr int kChunk = 16;  // rows per chunk

// Device status codes (same values as kda_status).
constexpr int32_t kStatusOk = 0;
constexpr int32_t kStatusBadSeqlens = 1;
constexpr int32_t kStatusTimeout = 7;

// Everything a forward launch needs; plain pointers and sizes.
struct FwdParams {
    const __nv_bfloat16* q;
    const __nv_bfloat16* k;
    const __nv_bfloat16* v;
    const float* g;
    const __nv_bfloat16* beta;
    const float* s0;      // [N][H][128][128] or nullptr (zero state)
    float* sfin;          // [N][H][128][128] or nullptr (not written)
    __nv_bfloat16* out;   // [T_total][H][128]
    const int32_t* cu;    // [N + 1] or nullptr (dense)
    int64_t T_total;
    int64_t dense_len;    // tokens per sequence when cu == nullptr
    int32_t N;
    int32_t H;
    float scale;
    int64_t wait_limit;   // iteration limit of bounded spin waits
    int32_t debug_flags;  // KDA_DEBUG_* bits (failure-path tests only)
    int32_t* status;      // device status word of this device
    // Segment launches (seg_len > 0): CTA row n' = b * nseg_used + s runs segment s of
    // dense sequence b, tokens [b*L + s*seg_len, b*L + min((s+1)*seg_len, L)), L = dense_len.
    int64_t seg_len;
    int32_t nseg_used;    // segments of each sequence covered by this launch
    int32_t nseg_total;   // segments of each sequence
    int32_t flags;        // kFlag* below
};

// Launch flags of the fused kernel.
constexpr int32_t kFlagNoOutput = 1;       // no output rows (summary runs)
constexpr int32_t kFlagZeroV = 2;          // treat v as zero (transition runs: U = 0)
constexpr int32_t kFlagIdentityS0 = 4;     // initial state = identity
constexpr int32_t kFlagFinalLastSeg = 8;   // write final state only for the last segment, at index b

// Token range [bos, eos) of sequence n; false (and the status word set) when
// cu_seqlens is malformed for this sequence.
__device__ __forceinline__ bool seq_range(const FwdParams& p, int n, int64_t& bos,
                                          int64_t& eos) {
    if (p.seg_len > 0) {
        const int b = n / p.nseg_used, sg = n % p.nseg_used;
        const int64_t base = (int64_t)b * p.dense_len;
        const int64_t a = (int64_t)sg * p.seg_len;
        bos = base + a;
        eos = base + (a + p.seg_len < p.dense_len ? a + p.seg_len : p.dense_len);
        return true;
    }
    if (p.cu == nullptr) {
        bos = (int64_t)n * p.dense_len;
        eos = bos + p.dense_len;
        return true;
    }
    bos = p.cu[n];
    eos = p.cu[n + 1];
    if ((n == 0 && bos != 0) || bos < 0 || eos < bos || eos > p.T_total) {
        atomicCAS(p.status, kStatusOk, kStatusBadSeqlens);
        return false;
    }
    return true;
}

// TMA descriptors of the [T_total][H][128] inputs, box {128, 1, 16} (one chunk of
// one head).  Encoded on the host, passed to kernels as __grid_constant__ params.
struct TensorMaps {
    CUtensorMap q, k, v, g;
    CUtensorMap out;  // output (TMA stores of full chunks)
};

// Launchers (return the launch error, cudaSuccess on success).
// Fused K1+K2 kernel over p.N x p.H rows (or the segment rows of a segment launch).
cudaError_t launch_serial(const FwdParams& p, const TensorMaps& maps, cudaStream_t stream);
// Segment merge: carry[b][0] = S0[b] (or 0), carry[b][s+1] = m[b][s] carry[b][s] + bs[b][s].
cudaError_t launch_merge(const float* m_seg, const float* b_seg, const float* s0, float* carries,
                         int32_t B, int32_t nseg, int32_t H, cudaStream_t stream);
size_t serial_smem_bytes();
int serial_block_threads();
const void* serial_kernel_symbol();
size_t merge_smem_bytes();
const void* merge_kernel_symbol();

}  // namespace kda
