// kda_merge.cu -- the "merge" step of segment-parallel prefill: the serial combine of
// per-segment summaries into the carry (state at each segment start).
//
// Segment pipeline (cuLA PR #103, FlashKDA prefill port with intra-card context
// parallelism, commit notes): a long sequence is cut into segments; K1 runs once, a
// pre_scan summarises every segment, the merge below chains the summaries, and a second
// K2 pass runs each segment from its carry.  Over one segment the state map is affine,
// S_end = m_seg S_start + b_seg, so
//     carry_0 = S_0 (or 0),   carry_{s+1} = m_seg[s] carry_s + b_seg[s].
// One CTA per (sequence, head, column block of the carry): the carry's columns are
// independent, so each CTA runs the whole serial chain over segments for its block.  The
// next segment's transition and summary block stream into a second shared-memory buffer
// (16-byte cp.async) while the current product runs, so a step of the chain waits on no
// global load.  The two halves of the CTA take the two halves of each product's K range
// (the upper half hands its partial sums over in shared memory), so sixteen warps hide
// the shared-memory load latency of a step.  The block width is the widest of 32 / 16 /
// 8 columns that still gives every SM a CTA, so that few heads spread over the GPU.
// fp32 throughout (the carries feed every later output of their segment).
#include "kda_internal.cuh"

namespace kda {
namespace {

constexpr int kMergeThreads = 512;              // two K halves of 256 threads
constexpr int kHalfThreads = kMergeThreads / 2;
constexpr int kMRow = kD + 4;  // padded row of a transition in shared memory

template <int kCols>
struct MergeShape {
    static constexpr int kColGroups = kCols / 4;                  // float4 columns
    static constexpr int kRowGroups = kHalfThreads / kColGroups;  // threads along rows
    static constexpr int kRowsPer = kD / kRowGroups;              // rows per thread
    static constexpr int kBRow = kCols + 4;                       // padded row of a block
    static constexpr int kMFloats = kD * kMRow;
    static constexpr int kBFloats = kD * kBRow;
    static constexpr int kPFloats = kHalfThreads * kRowsPer * 4;  // upper-half partials
    // two transitions, two summary blocks, the carry block, the partials
    static constexpr int kSmem = (2 * kMFloats + 3 * kBFloats + kPFloats) * 4;
};

__device__ __forceinline__ void cp_async16(float* sdst, const float* gsrc) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(sdst);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int kPending>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(kPending) : "memory");
}

template <int kCols>
__global__ void __launch_bounds__(kMergeThreads)
kda_merge_kernel(const float* __restrict__ m_seg, const float* __restrict__ b_seg,
                 const void* __restrict__ s0, int s0_bf16, float* __restrict__ carries, int B, int nseg,
                 int H, const int32_t* __restrict__ seg_start) {
    using S = MergeShape<kCols>;
    extern __shared__ __align__(16) float sm[];
    float* Ms = sm;                        // two transitions m[i][k], rows padded
    float* Bsm = sm + 2 * S::kMFloats;     // two summary blocks b[i][c]
    float* Cb = Bsm + 2 * S::kBFloats;     // carry block [k][c]
    float* Pp = Cb + S::kBFloats;          // partial sums of the upper K half
    const int tid = threadIdx.x;
    const int lo = tid % kHalfThreads, kh = tid / kHalfThreads;  // K half: keys 64 kh ..
    constexpr int kBlocks = kD / kCols;
    const int cb = blockIdx.x % kBlocks;
    const int h = (blockIdx.x / kBlocks) % H;
    const int b = blockIdx.x / (kBlocks * H);
    // Thread tile: rows rg + kRowGroups*a (a < kRowsPer), columns c0..c0+3 of the block.
    // A warp's rows are consecutive, so its float4 reads of a padded transition row fall
    // on distinct banks; its columns are consecutive float4s of one carry row.
    const int rg = lo / S::kColGroups;
    const int c0 = (lo % S::kColGroups) * 4;
    const size_t st = (size_t)kD * kD;
    // Dense: summaries [B][nseg-1][H], carries [B][nseg][H].  Varlen: every table indexed
    // by the global segment row g = seg_start[b] + s, sequence b owning its own count.
    size_t g0 = 0;
    int ns = nseg;
    if (seg_start) {
        g0 = (size_t)seg_start[b];
        ns = seg_start[b + 1] - seg_start[b];
    }
    if (ns <= 0) return;  // malformed cu_seqlens: the table is all zeros and nothing runs
    auto carry_at = [&](int s) {
        return carries + ((seg_start ? g0 + s : (size_t)b * nseg + s) * H + h) * st;
    };
    auto summary_at = [&](const float* base, int s) {
        return base + ((seg_start ? g0 + s : (size_t)b * (nseg - 1) + s) * H + h) * st;
    };
    auto prefetch = [&](int s, int buf) {
        const float* M = summary_at(m_seg, s);
        const float* Bs = summary_at(b_seg, s) + cb * kCols;
        float* Md = Ms + buf * S::kMFloats;
        float* Bd = Bsm + buf * S::kBFloats;
        for (int e = tid; e < kD * (kD / 4); e += kMergeThreads) {
            const int i = e / (kD / 4), j = e % (kD / 4);
            cp_async16(Md + i * kMRow + 4 * j, M + (size_t)i * kD + 4 * j);
        }
        for (int e = tid; e < kD * S::kColGroups; e += kMergeThreads) {
            const int i = e / S::kColGroups, j = e % S::kColGroups;
            cp_async16(Bd + i * S::kBRow + 4 * j, Bs + (size_t)i * kD + 4 * j);
        }
        cp_async_commit();
    };

    if (ns > 1) prefetch(0, 0);
    // carry_0
    for (int e = tid; e < kD * kCols; e += kMergeThreads) {
        const int k = e / kCols, c = e % kCols;
        const size_t i0 = ((size_t)b * H + h) * st + (size_t)k * kD + cb * kCols + c;
        const float v = s0 == nullptr ? 0.f
                        : s0_bf16     ? __bfloat162float(static_cast<const __nv_bfloat16*>(s0)[i0])
                                      : static_cast<const float*>(s0)[i0];
        Cb[k * S::kBRow + c] = v;
        carry_at(0)[(size_t)k * kD + cb * kCols + c] = v;
    }
    for (int s = 0; s + 1 < ns; ++s) {
        // Buffer (s+1)&1 was last read in step s-1, which ended on a barrier.
        if (s + 2 < ns) {
            prefetch(s + 1, (s + 1) & 1);
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();  // step s's buffers and the carry block written in step s-1
        const float* Mb = Ms + (s & 1) * S::kMFloats;
        const float* Bb = Bsm + (s & 1) * S::kBFloats;
        float acc[S::kRowsPer][4];
#pragma unroll
        for (int a = 0; a < S::kRowsPer; ++a) {
            float4 bv = make_float4(0.f, 0.f, 0.f, 0.f);
            if (kh == 0) bv = *reinterpret_cast<const float4*>(Bb + (rg + S::kRowGroups * a) * S::kBRow + c0);
            acc[a][0] = bv.x;
            acc[a][1] = bv.y;
            acc[a][2] = bv.z;
            acc[a][3] = bv.w;
        }
#pragma unroll 2
        for (int k = kh * (kD / 2); k < (kh + 1) * (kD / 2); k += 4) {
            float mm[S::kRowsPer][4];
#pragma unroll
            for (int a = 0; a < S::kRowsPer; ++a) {
                const float4 mv = *reinterpret_cast<const float4*>(Mb + (rg + S::kRowGroups * a) * kMRow + k);
                mm[a][0] = mv.x;
                mm[a][1] = mv.y;
                mm[a][2] = mv.z;
                mm[a][3] = mv.w;
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const float4 cv = *reinterpret_cast<const float4*>(Cb + (k + kk) * S::kBRow + c0);
#pragma unroll
                for (int a = 0; a < S::kRowsPer; ++a) {
                    acc[a][0] = fmaf(mm[a][kk], cv.x, acc[a][0]);
                    acc[a][1] = fmaf(mm[a][kk], cv.y, acc[a][1]);
                    acc[a][2] = fmaf(mm[a][kk], cv.z, acc[a][2]);
                    acc[a][3] = fmaf(mm[a][kk], cv.w, acc[a][3]);
                }
            }
        }
        if (kh == 1) {
#pragma unroll
            for (int a = 0; a < S::kRowsPer; ++a)
                *reinterpret_cast<float4*>(Pp + (a * kHalfThreads + lo) * 4) =
                    make_float4(acc[a][0], acc[a][1], acc[a][2], acc[a][3]);
        }
        __syncthreads();  // partials written; every read of the carry block and buffer s&1 done
        if (kh == 0) {
            float* out = carry_at(s + 1);
#pragma unroll
            for (int a = 0; a < S::kRowsPer; ++a) {
                const int i = rg + S::kRowGroups * a;
                const float4 pv = *reinterpret_cast<const float4*>(Pp + (a * kHalfThreads + lo) * 4);
                const float4 o = make_float4(acc[a][0] + pv.x, acc[a][1] + pv.y, acc[a][2] + pv.z,
                                             acc[a][3] + pv.w);
                *reinterpret_cast<float4*>(Cb + i * S::kBRow + c0) = o;
                *reinterpret_cast<float4*>(out + (size_t)i * kD + cb * kCols + c0) = o;
            }
        }
    }
}

template <int kCols>
cudaError_t merge_set_smem() {
    return cudaFuncSetAttribute(kda_merge_kernel<kCols>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                MergeShape<kCols>::kSmem);
}

template <int kCols>
cudaError_t merge_launch(const float* m_seg, const float* b_seg, const void* s0, int s0_bf16, float* carries,
                         int32_t B, int32_t nseg, int32_t H, cudaStream_t stream,
                         const int32_t* seg_start) {
    const long long blocks = (long long)B * H * (kD / kCols);
    kda_merge_kernel<kCols><<<(unsigned)blocks, kMergeThreads, MergeShape<kCols>::kSmem, stream>>>(
        m_seg, b_seg, s0, s0_bf16, carries, B, nseg, H, seg_start);
    return cudaGetLastError();
}

}  // namespace

cudaError_t merge_init() {
    cudaError_t e;
    if ((e = merge_set_smem<32>()) || (e = merge_set_smem<16>()) || (e = merge_set_smem<8>())) return e;
    return cudaSuccess;
}

int merge_block_cols(int32_t B, int32_t H, int sm_count) {
    const long long heads = (long long)B * H;
    if (heads * (kD / 32) >= sm_count) return 32;
    if (heads * (kD / 16) >= sm_count) return 16;
    return 8;
}

cudaError_t launch_merge(const float* m_seg, const float* b_seg, const void* s0, int s0_bf16, float* carries,
                         int32_t B, int32_t nseg, int32_t H, int sm_count, cudaStream_t stream,
                         const int32_t* seg_start) {
    if ((long long)B * H == 0) return cudaSuccess;
    switch (merge_block_cols(B, H, sm_count)) {
        case 32: return merge_launch<32>(m_seg, b_seg, s0, s0_bf16, carries, B, nseg, H, stream, seg_start);
        case 16: return merge_launch<16>(m_seg, b_seg, s0, s0_bf16, carries, B, nseg, H, stream, seg_start);
        default: return merge_launch<8>(m_seg, b_seg, s0, s0_bf16, carries, B, nseg, H, stream, seg_start);
    }
}

// One CTA: validate cu_seqlens (cu[0] = 0, non-decreasing, cu[N] <= T_total), then an
// exclusive scan of max(1, ceil(len / seg_len)).  On malformed input the status word is
// set and the table is all zeros, so every segment row of the following launches exits.
__global__ void __launch_bounds__(1024)
kda_segment_table_kernel(const int32_t* __restrict__ cu, int N, long long T_total, long long seg_len,
                         int32_t* __restrict__ seg_start, int32_t* status) {
    __shared__ int32_t warp_sums[32];
    __shared__ int32_t carry;
    __shared__ int bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        carry = 0;
        bad = 0;
    }
    __syncthreads();
    for (int n = tid; n < N; n += blockDim.x) {
        const long long a = cu[n], e = cu[n + 1];
        if ((n == 0 && a != 0) || a < 0 || e < a || e > T_total) bad = 1;
    }
    __syncthreads();
    if (bad) {
        if (tid == 0) atomicCAS(status, kStatusOk, kStatusBadSeqlens);
        for (int n = tid; n <= N; n += blockDim.x) seg_start[n] = 0;
        return;
    }
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int32_t cnt = 0;
        if (n < N) {
            const long long len = (long long)cu[n + 1] - cu[n];
            const long long c = (len + seg_len - 1) / seg_len;
            cnt = (int32_t)(c > 1 ? c : 1);
        }
        int32_t incl = cnt;  // inclusive warp scan
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const int32_t o = __shfl_up_sync(0xffffffffu, incl, d);
            if (lane >= d) incl += o;
        }
        if (lane == 31) warp_sums[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            int32_t w = lane < (int)(blockDim.x >> 5) ? warp_sums[lane] : 0;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int32_t o = __shfl_up_sync(0xffffffffu, w, d);
                if (lane >= d) w += o;
            }
            warp_sums[lane] = w;  // inclusive over warps
        }
        __syncthreads();
        const int32_t before = carry + (warp > 0 ? warp_sums[warp - 1] : 0) + incl - cnt;
        if (n < N) seg_start[n] = before;
        __syncthreads();
        if (tid == 0) carry += warp_sums[(blockDim.x >> 5) - 1];
        __syncthreads();
    }
    if (tid == 0) seg_start[N] = carry;
}

cudaError_t launch_segment_table(const int32_t* cu, int32_t N, int64_t T_total, int64_t seg_len,
                                 int32_t* seg_start, int32_t* status, cudaStream_t stream) {
    kda_segment_table_kernel<<<1, 1024, 0, stream>>>(cu, N, (long long)T_total, (long long)seg_len,
                                                    seg_start, status);
    return cudaGetLastError();
}

}  // namespace kda
