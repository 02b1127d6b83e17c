// mma_peak.cu -- dense tensor-core throughput of tcgen05.mma on the GPU at
// hand: the denominator of the prefill scoring kernel's roofline.
//
// Every CTA (one per SM) keeps an A tile (128 rows) and a B tile (256 rows)
// of 128-byte K-major rows resident in shared memory (128-byte swizzle) and
// one thread issues `iters` rounds of four back-to-back MMAs (M = 128,
// N = 256, K = 32 bytes of the row per MMA) accumulating into a 256-column
// TMEM tile, then commits once and waits (bounded) for them.  Nothing is
// loaded from memory inside the timed loop, so the time is the tensor pipe's.
//   kind::f8f6f4 (e4m3 x e4m3): K = 32 per MMA, 2 * 128 * 256 * 32 flops;
//   kind::f16    (bf16 x bf16): K = 16 per MMA, 2 * 128 * 256 * 16 flops.
// The bf16 figure checks the method against a cuBLAS bf16 GEMM.
#include <cuda_runtime.h>

#include "common.cuh"

namespace {

using namespace dsaidx;

constexpr int kPeakM = 128;
constexpr int kPeakN = 256;
constexpr int kPeakThreads = 128;
constexpr int kPeakSmem = 16384 + 32768 + 1024 + 1024;   // A, B, barrier, alignment

template <bool kFp8>
__global__ void __launch_bounds__(kPeakThreads, 1) mma_peak_kernel(long long iters, int32_t* status, float* out) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* a = smem;                   // 128 rows x 128 bytes
    uint8_t* b = smem + 16384;           // 256 rows x 128 bytes
    uint64_t* bar = reinterpret_cast<uint64_t*>(smem + 16384 + 32768);
    uint32_t* tbase = reinterpret_cast<uint32_t*>(bar + 1);
    const int tid = threadIdx.x;
    // small finite operands (e4m3 0x30 = 0.5 in every byte; bf16 0.5)
    const uint32_t pat = kFp8 ? 0x30303030u : 0x3F003F00u;
    for (int i = tid; i < (16384 + 32768) / 16; i += kPeakThreads)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(pat, pat, pat, pat);
    fence_proxy_async_smem();
    if (tid < 32) {
        tmem_alloc(tbase, kPeakN);
        tmem_relinquish();
    }
    if (tid == 32) {
        mbar_init(bar, 1);
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t d = *tbase;
    if (tid == 0) {
        constexpr uint32_t idesc = idesc_make(kFp8, kPeakM, kPeakN);
        const uint32_t ab = smem_u32(a), bb = smem_u32(b);
        for (long long it = 0; it < iters; ++it) {
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const uint64_t ad = sdesc_sw128(ab + 32 * k), bd = sdesc_sw128(bb + 32 * k);
                if constexpr (kFp8) mma_fp8(d, ad, bd, idesc, (it | k) != 0 ? 1u : 0u);
                else mma_bf16(d, ad, bd, idesc, (it | k) != 0 ? 1u : 0u);
            }
        }
        mma_commit(bar);
        mbar_wait(bar, 0u, status, nullptr);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (out != nullptr && blockIdx.x == 0) {
        // the accumulator's row `tid`, every 16th column: each warp reads its 32 TMEM lanes
        for (int c = 0; c < kPeakN; c += 16) {
            float v[16];
            tmem_ld16(d + (static_cast<uint32_t>(32 * (tid >> 5)) << 16) + static_cast<uint32_t>(c), v);
            out[tid * (kPeakN / 16) + c / 16] = v[c / 16 % 16];
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (tid < 32) tmem_dealloc(d, kPeakN);
}

}  // namespace

// Runs `launches` launches of the kernel (one CTA per SM, `iters` rounds of 4
// MMAs each) back to back on the current device and returns the dense
// throughput in TFLOP/s in *tflops and the elapsed milliseconds in *ms.
// fp8 != 0: kind::f8f6f4 e4m3; 0: kind::f16 bf16.  A check launch of 8
// rounds first reads 2048 accumulator entries back: every one must be
// 8 * 4 * K * 0.25 (all operands 0.5).  Returns 0 on success, 1 on a CUDA
// error, 2 when a wait ran out (status word set), 3 when the check fails.
extern "C" int mma_peak_run(int fp8, long long iters, int launches, double* tflops, double* ms) {
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 1;
    auto kern = fp8 ? mma_peak_kernel<true> : mma_peak_kernel<false>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kPeakSmem) != cudaSuccess) return 1;
    int32_t* status = nullptr;
    if (cudaMalloc(&status, sizeof(int32_t)) != cudaSuccess) return 1;
    cudaMemset(status, 0, sizeof(int32_t));
    cudaEvent_t e0, e1;
    cudaEventCreate(&e0);
    cudaEventCreate(&e1);
    float* chk = nullptr;
    if (cudaMalloc(&chk, sizeof(float) * kPeakThreads * (kPeakN / 16)) != cudaSuccess) return 1;
    kern<<<sms, kPeakThreads, kPeakSmem>>>(8, status, chk);   // warm-up and check
    float host[kPeakThreads * (kPeakN / 16)];
    bool good = cudaMemcpy(host, chk, sizeof(host), cudaMemcpyDeviceToHost) == cudaSuccess;
    const float expect = 8.0f * 4.0f * (fp8 ? 32.0f : 16.0f) * 0.25f;
    for (int i = 0; good && i < kPeakThreads * (kPeakN / 16); ++i) good = host[i] == expect;
    cudaFree(chk);
    cudaEventRecord(e0);
    for (int l = 0; l < launches; ++l) kern<<<sms, kPeakThreads, kPeakSmem>>>(iters, status, nullptr);
    cudaEventRecord(e1);
    int rc = cudaEventSynchronize(e1) == cudaSuccess && cudaGetLastError() == cudaSuccess ? 0 : 1;
    float t = 0.0f;
    cudaEventElapsedTime(&t, e0, e1);
    int32_t st = 0;
    cudaMemcpy(&st, status, sizeof(int32_t), cudaMemcpyDeviceToHost);
    if (rc == 0 && st != 0) rc = 2;
    if (rc == 0 && !good) rc = 3;
    const double flop_per_mma = 2.0 * kPeakM * kPeakN * (fp8 ? 32.0 : 16.0);
    const double flops = flop_per_mma * 4.0 * static_cast<double>(iters) * sms * launches;
    *ms = t;
    *tflops = t > 0.0f ? flops / (t * 1e-3) / 1e12 : 0.0;
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    cudaFree(status);
    return rc;
}
