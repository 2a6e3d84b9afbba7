// Host-side pieces of the C ABI: defaults, version, per-thread error text.
#include <cmath>
#include <mutex>

#include "common.cuh"

namespace csa2 {

static thread_local std::string g_last_error;

void set_error(const std::string& msg) { g_last_error = msg; }

int fail(int code, const std::string& msg) {
    g_last_error = msg;
    return code;
}

int check_launch(const char* what) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess)
        return fail(CSA2_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
    return CSA2_OK;
}

int ensure_loaded() {
    static std::mutex mu;
    static uint64_t done = 0;  // bit d: device d loaded
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return check_launch("device");
    if (dev < 0 || dev >= 64) return CSA2_OK;
    std::lock_guard<std::mutex> g(mu);
    if ((done >> dev) & 1u) return CSA2_OK;
    cudaError_t (*lists[])() = {preload_compress, preload_index, preload_index_shared,
                                preload_select, preload_attn, preload_attn_tc, preload_peak};
    for (auto f : lists) {
        const cudaError_t e = f();
        if (e != cudaSuccess) {
            cudaGetLastError();
            return fail(CSA2_ERR_CUDA, std::string("loading the kernels: ") + cudaGetErrorString(e));
        }
    }
    done |= 1ull << dev;
    return CSA2_OK;
}

}  // namespace csa2

extern "C" void csa2_default_params(csa2_params* p) {
    if (!p) return;
    p->heads = csa2::kH;
    p->head_dim = csa2::kD;
    p->index_heads = csa2::kHi;
    p->index_dim = csa2::kDi;
    p->window = csa2::kW;
    p->block_size = csa2::kBlk;
    p->topk_blocks = csa2::kKb;
    p->topk_pos = csa2::kKp;
    p->compress_ratio = 2;
    p->kv_format = CSA2_NVFP4;
    p->win_format = CSA2_E4M3;
    p->q_format = CSA2_BF16;
    p->softmax_scale = 1.0f / std::sqrt((float)csa2::kD);
    p->win_layout = CSA2_WIN_RING;
    p->max_ctas = 0;
    p->rope_dim = 0;
    p->rope_theta = 160000.0f;
    p->rope_factor = 16.0f;
    p->rope_orig_len = 65536.0f;
    p->rope_beta_fast = 32.0f;
    p->rope_beta_slow = 1.0f;
}

extern "C" int csa2_trace_attach(int32_t* record) {
    cudaError_t (*setters[])(int32_t*) = {csa2::trace_set_compress, csa2::trace_set_index,
                                          csa2::trace_set_select, csa2::trace_set_attn_tc};
    if (const int rc = csa2::ensure_loaded()) return rc;
    for (auto f : setters)
        if (f(record) != cudaSuccess) return csa2::check_launch("trace_attach");
    return CSA2_OK;
}

extern "C" int csa2_version(void) { return 300; }

extern "C" const char* csa2_last_error(void) { return csa2::g_last_error.c_str(); }
