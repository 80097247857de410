// tcgen05_probe.cu -- test-only check of the tcgen05 building blocks used by the
// library (shared-memory matrix descriptors of the no-swizzle K-major layout and of the
// 128-byte-swizzled M-major layout, the bf16 A operand held in TMEM, TMEM loads), on
// problems whose products the test recomputes on the host.  One CTA, 128 threads.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kda_ptx.cuh"

using namespace kda::ptx;

namespace {
constexpr uint32_t kLboK = 128, kSboA = 2048, kSboB2 = 256;

__device__ uint32_t kmajor_off(int row, int k, uint32_t lbo, uint32_t sbo) {
    return (row / 8) * sbo + (k / 8) * lbo + (row % 8) * 16 + (k % 8) * 2;
}

__global__ void __launch_bounds__(128, 1)
probe_kernel(const uint16_t* A, const uint16_t* B1, const uint16_t* B2, float* D1_ss,
             float* D1_ts, float* D2, int32_t* err, int64_t limit) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* a_sm = smem;                  // 128 x 128, 32 KiB
    unsigned char* b1_sm = smem + 32768;         // 32 x 128, 8 KiB
    unsigned char* b2_sm = smem + 40960;         // 128 x 16, 4 KiB
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid / 32;

    for (int e = tid; e < 128 * 128; e += 128) {
        const int m = e / 128, k = e % 128;
        *reinterpret_cast<uint16_t*>(a_sm + kmajor_off(m, k, kLboK, kSboA)) = A[e];
    }
    for (int e = tid; e < 32 * 128; e += 128) {
        const int n = e / 128, k = e % 128;
        *reinterpret_cast<uint16_t*>(b1_sm + kmajor_off(n, k, kLboK, kSboA)) = B1[e];
    }
    for (int e = tid; e < 128 * 16; e += 128) {
        const int n = e / 16, k = e % 16;
        *reinterpret_cast<uint16_t*>(b2_sm + kmajor_off(n, k, kLboK, kSboB2)) = B2[e];
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base), 256);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    const uint32_t t_d1ss = tbase + 0, t_d1ts = tbase + 32, t_a = tbase + 64, t_d2 = tbase + 128;

    // Row m of A into TMEM as packed bf16 pairs (low half = even k).
    uint32_t packed[64];
    for (int c = 0; c < 64; ++c)
        packed[c] = (uint32_t)A[tid * 128 + 2 * c] | ((uint32_t)A[tid * 128 + 2 * c + 1] << 16);
    tmem_st32(t_a + lane_base, packed);
    tmem_st32(t_a + lane_base + 32, packed + 32);
    tmem_wait_st();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();

    if (tid == 0) {
        const uint32_t a0 = smem_u32(a_sm), b10 = smem_u32(b1_sm), b20 = smem_u32(b2_sm);
        for (int kk = 0; kk < 8; ++kk)
            mma_ss(t_d1ss, sdesc(a0 + kk * 2 * kLboK, kLboK, kSboA),
                   sdesc(b10 + kk * 2 * kLboK, kLboK, kSboA), idesc_bf16(128, 32), kk > 0);
        for (int kk = 0; kk < 8; ++kk)
            mma_ts(t_d1ts, t_a + kk * 8, sdesc(b10 + kk * 2 * kLboK, kLboK, kSboA),
                   idesc_bf16(128, 32), kk > 0);
        mma_ts(t_d2, t_a, sdesc(b20, kLboK, kSboB2), idesc_bf16(128, 128), 0);
        tc_commit(smem_u32(&bar));
    }
    const bool ok = mbar_wait(smem_u32(&bar), 0, limit);
    if (!ok) atomicExch(err, 7);
    tc_fence_after();
    if (ok) {
        uint32_t r[32];
        tmem_ld32(t_d1ss + lane_base, r);
        tmem_wait_ld_regs<32>(r);
        for (int c = 0; c < 32; ++c) D1_ss[tid * 32 + c] = __uint_as_float(r[c]);
        tmem_ld32(t_d1ts + lane_base, r);
        tmem_wait_ld_regs<32>(r);
        for (int c = 0; c < 32; ++c) D1_ts[tid * 32 + c] = __uint_as_float(r[c]);
        for (int q = 0; q < 4; ++q) {
            tmem_ld32(t_d2 + lane_base + 32 * q, r);
            tmem_wait_ld_regs<32>(r);
            for (int c = 0; c < 32; ++c) D2[tid * 128 + 32 * q + c] = __uint_as_float(r[c]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 256);
}
// A operand stored M-major (MN-major) with the 128-byte swizzle, as a TMA load with
// CU_TENSOR_MAP_SWIZZLE_128B writes a [K][M] bf16 tile in two boxes of 64 M-columns:
// box h (M columns 64h .. 64h+63) at byte 2048h, row k (K index) at 128k within it, the
// 16-byte chunk index of a row XORed with k % 8.  Descriptor: LBO = 2048 (between the
// two 64-column boxes), SBO = 1024 (between the two 8-row K groups), swizzle mode 2.
// D[m][n] = sum_k V[k][m] B[n][k] for M = 128, N = 16, K = 16, B K-major without swizzle.
__global__ void __launch_bounds__(128, 1)
probe_mn_sw128(const uint16_t* V, const uint16_t* B, float* D, int32_t* err, int64_t limit) {
    extern __shared__ __align__(1024) unsigned char smem[];
    unsigned char* v_sm = smem;          // 2 boxes x 16 rows x 128 B = 4 KiB
    unsigned char* b_sm = smem + 4096;   // 16 x 16, K-major
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int tid = threadIdx.x, warp = tid / 32;
    if (tid == 0 && (smem_u32(v_sm) & 1023u) != 0) atomicExch(err, 9);  // the swizzle needs 1 KiB alignment
    for (int e = tid; e < 16 * 128; e += 128) {
        const int k = e / 128, m = e % 128;
        const int box = m / 64, byte = (m % 64) * 2;
        const int chunk = (byte / 16) ^ (k % 8);
        *reinterpret_cast<uint16_t*>(v_sm + box * 2048 + k * 128 + chunk * 16 + byte % 16) = V[e];
    }
    for (int e = tid; e < 16 * 16; e += 128) {
        const int n = e / 16, k = e % 16;
        *reinterpret_cast<uint16_t*>(b_sm + kmajor_off(n, k, kLboK, kSboB2)) = B[e];
    }
    if (tid == 0) {
        mbar_init(smem_u32(&bar), 1);
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(&tmem_base), 32);
        tmem_relinquish();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tbase = tmem_base;
    const uint32_t lane_base = (uint32_t)(32 * warp) << 16;
    if (tid == 0) {
        const uint64_t adesc = sdesc(smem_u32(v_sm), 2048, 1024) | ((uint64_t)2 << 61);
        mma_ss(tbase, adesc, sdesc(smem_u32(b_sm), kLboK, kSboB2), idesc_bf16(128, 16) | (1u << 15), 0);
        tc_commit(smem_u32(&bar));
    }
    const bool ok = mbar_wait(smem_u32(&bar), 0, limit);
    if (!ok) atomicExch(err, 7);
    tc_fence_after();
    if (ok) {
        uint32_t r[16];
        tmem_ld16(tbase + lane_base, r);
        tmem_wait_ld_regs<16>(r);
        for (int c = 0; c < 16; ++c) D[tid * 16 + c] = __uint_as_float(r[c]);
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 0) tmem_dealloc(tbase, 32);
}
}  // namespace

extern "C" int tcgen05_probe_mn_sw128(const uint16_t* V, const uint16_t* B, float* D, int32_t* err) {
    const int smem = 8192;
    probe_mn_sw128<<<1, 128, smem>>>(V, B, D, err, 1 << 22);
    return (int)cudaDeviceSynchronize();
}

extern "C" int tcgen05_probe(const uint16_t* A, const uint16_t* B1, const uint16_t* B2,
                             float* D1_ss, float* D1_ts, float* D2, int32_t* err) {
    const int smem = 45056;
    cudaFuncSetAttribute(probe_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    probe_kernel<<<1, 128, smem>>>(A, B1, B2, D1_ss, D1_ts, D2, err, 1 << 22);
    cudaError_t e = cudaDeviceSynchronize();
    return (int)e;
}
