// Measurement aid (no counterpart in the pages): the rate of the block-scaled
// FP4 tensor-core MMA that the prefill Indexer issues (index_shared.cu), so the
// Indexer's throughput can be stated as a fraction of what this GPU's tensor
// pipe reaches with the same instruction. Every CTA keeps one A tile (128 rows)
// and one B tile (128 rows) of E2M1 codes with the 64-byte swizzle, and their
// E4M3 scale factors copied into TMEM, and one thread issues `iters` pairs of
// tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M = 128, N = 128, K = 64
// each, so K = 128 per pair) back to back into one TMEM accumulator. Operands
// are fixed pseudo-random codes and unit scales (the values do not matter).
#include "common.cuh"
#include "sm100.cuh"

namespace csa2 {
namespace {
using namespace sm100;

constexpr int kPeakThreads = 128;
constexpr int kRows = 128;           // M = N = 128
constexpr int kTileBytes = kRows * 64;  // 128 rows x 128 E2M1 codes
constexpr uint32_t kPeakCols = 256;  // D (128 columns) + scale factors
constexpr uint32_t kColSFA = 128, kColSFB = 136;
// kind::mxf4nvf4, A and B E2M1, K-major, N = 128 (N>>3 in bits 17..22), UE4M3
// scales, M = 128 (M>>4 in bits 24..28): the prefill Indexer's descriptor.
constexpr uint32_t kPeakIdesc = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);

struct PeakShared {
    uint8_t a[kTileBytes];  // 1024-aligned (the 64-byte swizzle repeats every 512 bytes)
    uint8_t b[kTileBytes];
    uint8_t sfa[1024];      // two 512-byte scale-factor atoms (K 0..63, 64..127)
    uint8_t sfb[1024];
    uint64_t done;
    uint32_t tmem_base;
};
constexpr int kPeakSmem = (int)sizeof(PeakShared) + 1024;

__global__ void __launch_bounds__(kPeakThreads, 1) k_fp4_mma_peak(int iters, int32_t* dev_status) {
    extern __shared__ uint8_t smem_raw[];
    PeakShared& sh =
        *reinterpret_cast<PeakShared*>(smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u));
    const int tid = threadIdx.x, warp = tid >> 5;
    // operands: codes from a multiplicative hash of the byte offset, scales 1.0 (0x38)
    for (int i = tid; i < kTileBytes / 4; i += kPeakThreads) {
        reinterpret_cast<uint32_t*>(sh.a)[i] = (uint32_t)i * 2654435761u;
        reinterpret_cast<uint32_t*>(sh.b)[i] = ((uint32_t)i ^ 0x5bd1e995u) * 2246822519u;
    }
    for (int i = tid; i < 1024 / 4; i += kPeakThreads) {
        reinterpret_cast<uint32_t*>(sh.sfa)[i] = 0x38383838u;
        reinterpret_cast<uint32_t*>(sh.sfb)[i] = 0x38383838u;
    }
    if (tid == 0) {
        mbar_init(&sh.done, 1);
        fence_mbar_init();
    }
    fence_proxy_async_smem();  // the operands above are read by the tensor core
    if (warp == 0) {
        tmem_alloc(&sh.tmem_base, kPeakCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = sh.tmem_base;
    bool ok = true;
    if (warp == 0) {
        if (elect_one()) {
            tmem_cp_32x128b_x4(tmem + kColSFA, smem_desc(smem_u32(sh.sfa), 128, 128, kLayoutNone));
            tmem_cp_32x128b_x4(tmem + kColSFA + 4, smem_desc(smem_u32(sh.sfa) + 512, 128, 128, kLayoutNone));
            tmem_cp_32x128b_x4(tmem + kColSFB, smem_desc(smem_u32(sh.sfb), 128, 128, kLayoutNone));
            tmem_cp_32x128b_x4(tmem + kColSFB + 4, smem_desc(smem_u32(sh.sfb) + 512, 128, 128, kLayoutNone));
            const uint64_t dA = smem_desc(smem_u32(sh.a), 16, 512, kLayoutSw64);
            const uint64_t dB = smem_desc(smem_u32(sh.b), 16, 512, kLayoutSw64);
            for (int i = 0; i < iters; ++i) {
                mma_mxf4nvf4(tmem, dA, dB, kPeakIdesc, tmem + kColSFA, tmem + kColSFB, i > 0 ? 1u : 0u);
                mma_mxf4nvf4(tmem, dA + 2, dB + 2, kPeakIdesc, tmem + kColSFA + 4, tmem + kColSFB + 4, 1u);
            }
            // arrives once every copy and MMA above has completed
            tc_commit(&sh.done);
        }
        __syncwarp();
        ok = mbar_wait_drain(&sh.done, 0);
        if (!ok && (tid & 31) == 0) raise_status(dev_status, CSA2_DEV_TIMEOUT);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 0) tmem_dealloc(tmem, kPeakCols);
}

}  // namespace

cudaError_t preload_peak() { return preload_kernel(k_fp4_mma_peak, kPeakSmem); }

}  // namespace csa2

using namespace csa2;

extern "C" int csa2_fp4_mma_peak(int ctas, int iters, int32_t* dev_status, void* stream) {
    if (ctas <= 0 || ctas > 65535 || iters <= 0 || iters > (1 << 22))
        return fail(CSA2_ERR_INVALID_ARG, "fp4_mma_peak: ctas in [1, 65535], iters in [1, 2^22]");
    if (const int rc = ensure_loaded()) return rc;
    k_fp4_mma_peak<<<ctas, kPeakThreads, kPeakSmem, static_cast<cudaStream_t>(stream)>>>(iters,
                                                                                        dev_status);
    return check_launch("fp4_mma_peak");
}
