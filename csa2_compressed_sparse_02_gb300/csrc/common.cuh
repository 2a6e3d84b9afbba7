// Internal helpers shared by the CSA2 kernels (sm_103a). Not part of the ABI.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <string>

#include "../../include/csa2.h"

namespace csa2 {

// Pages' sizes the kernels are specialised for ("CSA2稀疏注意力、384专家MoE与1M上下文"
// config walkthrough §2.1, §一; "DeepSeek-V4.1-Flash-NVFP4" §3.1-§3.3).
constexpr int kD = 512;       // KV latent dim
constexpr int kH = 64;        // query heads
constexpr int kHi = 32;       // index heads
constexpr int kDi = 128;      // index head dim
constexpr int kW = 128;       // window slots
constexpr int kBlk = 8;       // candidate block size
constexpr int kKb = 2048;     // blocks kept
constexpr int kKp = 512;      // positions kept
constexpr int kGroup = 16;    // NVFP4 group

void set_error(const std::string& msg);
int fail(int code, const std::string& msg);
int check_launch(const char* what);

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Loads a kernel's code now (a CUDA runtime that loads modules lazily would
// otherwise do it at the first launch or attribute call) and, when it asks
// for more than 48 KB of shared memory, sets that limit.
template <typename K>
inline cudaError_t preload_kernel(K* k, int smem = 0) {
    cudaFuncAttributes at;
    cudaError_t e = cudaFuncGetAttributes(&at, reinterpret_cast<const void*>(k));
    if (e == cudaSuccess && smem > 48 * 1024)
        e = cudaFuncSetAttribute(reinterpret_cast<const void*>(k),
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    return e;
}

// Every kernel of the library loaded and its attributes set on the current
// device, once per device, before the first launch of any of them. Returns
// CSA2_OK or CSA2_ERR_CUDA (text in csa2_last_error). Each translation unit
// contributes its own preload_* list.
int ensure_loaded();
cudaError_t preload_compress();
cudaError_t preload_index();
cudaError_t preload_index_shared();
cudaError_t preload_select();
cudaError_t preload_attn();
cudaError_t preload_attn_tc();
cudaError_t preload_peak();

// Single-layer sparse attention (csa2_sparse_attn, quantised formats) on the
// tcgen05 kernel of sparse_attn_tc.cu with the even split schedule; the
// workspace holds that schedule's partial results (sparse_attn_tc_ws_bytes),
// 256-byte aligned; its completion counts are zeroed on the stream first.
size_t sparse_attn_tc_ws_bytes(const csa2_params* p, int B);
int sparse_attn_tc_single(const char* name, const csa2_params* p, int B, const void* q,
                          const float* sink, const void* const* win, const int32_t* n_tokens,
                          const void* const* comp, const uint8_t* const* comp_scales,
                          const int32_t* idx, void* out, void* workspace, size_t ws_bytes,
                          int32_t* dev_status, void* stream);

// ---- launch trace (diagnostics; off unless csa2_trace_attach set a record).
// Every translation unit has its own copy of the record pointer. When set, CTA 0
// thread 0 of the traced kernels writes {kernel id, launch number} into record
// words 0-1 at its start and into words 2-3 when it finishes: plain posted stores
// to host-mapped memory (no fence: nothing waits for them), which the host can
// read after an error has ended the context. Kernels launched programmatically may
// start while the one ahead still runs: the record then holds whichever wrote last,
// and the launch number (a plain increment) may repeat across such a pair.
enum TraceKernel { kTraceCompress = 1, kTraceIndex = 2, kTraceSelect = 3, kTraceAttn = 4 };
namespace {
__device__ int32_t* g_trace = nullptr;
__device__ int32_t g_trace_seq = 0;
}  // namespace
__device__ __forceinline__ bool trace_lead() {
    return blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0;
}
__device__ __forceinline__ void trace_start(int id) {
    volatile int32_t* t = g_trace;
    if (t && trace_lead()) {
        const int32_t n = ++g_trace_seq;
        t[1] = n;
        t[0] = id;
    }
}
__device__ __forceinline__ void trace_end(int id) {
    volatile int32_t* t = g_trace;
    if (t && trace_lead()) {
        t[3] = g_trace_seq;
        t[2] = id;
    }
}
// Sets this translation unit's record pointer (NULL detaches).
#define CSA2_TRACE_SETTER(fn) \
    cudaError_t fn(int32_t* rec) { return cudaMemcpyToSymbol(g_trace, &rec, sizeof(rec)); }
cudaError_t trace_set_compress(int32_t* rec);
cudaError_t trace_set_index(int32_t* rec);
cudaError_t trace_set_select(int32_t* rec);
cudaError_t trace_set_attn_tc(int32_t* rec);

// Raise a status bit on the device (NULL status pointer = ignore).
__device__ __forceinline__ void raise_status(int32_t* st, int bit) {
    if (st) atomicOr(st, bit);
}

// E2M1 code of y: round to nearest, ties to the even code, |y| > 6 -> 6, sign
// bit from y. Thresholds are the midpoints of the E2M1 grid
// {0, .5, 1, 1.5, 2, 3, 4, 6}; at a midpoint the code with mantissa bit 0 wins,
// hence the alternation of > and >=.
__device__ __forceinline__ uint32_t e2m1_code_rne(float y) {
    float a = fabsf(y);
    uint32_t c = (a > 0.25f) + (a >= 0.75f) + (a > 1.25f) + (a >= 1.75f) + (a > 2.5f) +
                 (a >= 3.5f) + (a > 5.0f);
    return c | ((__float_as_uint(y) >> 28) & 8u);
}

// E4M3 byte of a float (hardware convert: RNE, saturating to +-448).
__device__ __forceinline__ uint8_t e4m3_byte(float x) {
    return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

// Value of an E4M3 byte (exact).
__device__ __forceinline__ float e4m3_value(uint8_t b) {
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)b, __NV_E4M3);
    return __half2float(__half(h));
}

// Two E2M1 codes (one byte, element 0 in the low nibble) -> two halves, exact.
__device__ __forceinline__ uint32_t e2m1x2_to_half2(uint32_t byte) {
    uint32_t out;
    asm("{\n .reg .b8 t;\n cvt.u8.u32 t, %1;\n cvt.rn.f16x2.e2m1x2 %0, t;\n}"
        : "=r"(out) : "r"(byte));
    return out;
}

// Order-preserving u32 key of an fp32 score (larger value -> larger key;
// -0 is folded onto +0 so that equal values tie).
__device__ __forceinline__ uint32_t score_key(float x) {
    uint32_t u = __float_as_uint(x + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

}  // namespace csa2

#define CSA2_CHECK_PARAMS(p)                                                    \
    do {                                                                        \
        if (!(p)) return csa2::fail(CSA2_ERR_INVALID_ARG, "params is NULL");    \
    } while (0)
