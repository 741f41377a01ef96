// fp_select_noalloc: the Stage 1 call for callers that cannot allocate device
// memory. Some callers have no way to obtain a scratch buffer: a plugin that
// an inference engine hands only its input and output tensors, or a caller on
// a path where cudaMalloc is not allowed because it can synchronise the device
// and stall other work. This entry point runs exactly the kernels of
// fp_select but takes its scratch from a fixed array compiled into the
// library, so the caller passes only inputs and outputs.
//
// The array is a file-scope device variable of kNoAllocScratchBytes (16 MiB).
// Every GPU that loads the library holds those bytes until the process exits.
// All calls share it and it keeps the last call's contents, so calls whose
// work overlaps on the GPU (on two streams, or from two host threads without
// ordering) race on it and must be serialised by the caller.
#include <mutex>
#include <stdio.h>

#include "fp_internal.cuh"

namespace fp {
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(16) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code may not use this name as a device address
// (on the host it only stands for the symbol); it asks the runtime for the
// address with cudaGetSymbolAddress instead.
static __device__ __align__(256) char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_mu;
char *g_scratch_ptr[kMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (the first call on each device does it, with that device current).
fp_status scratch_address(char **out) {
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        fprintf(stderr, "libfp: cudaGetDevice failed: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return FP_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess || !ptr) {
            fprintf(stderr, "libfp: cudaGetSymbolAddress of the static scratch failed: %s\n",
                    cudaGetErrorString(e));
            return FP_ERR_CUDA;
        }
        g_scratch_ptr[dev] = static_cast<char *>(ptr);
    }
    *out = g_scratch_ptr[dev];
    return FP_OK;
}

}  // namespace
}  // namespace fp

using namespace fp;

extern "C" fp_status fp_select_noalloc(const fp_problem *p, const void *q, const void *k_pages,
                                       const void *v_pages, float alpha, int32_t sink_blocks,
                                       int32_t window_blocks, int32_t *csr_cu, int32_t *csr_idx,
                                       int64_t csr_idx_capacity, float *kbar, float *vbar, void *kbar_op,
                                       void *vbar_op, int32_t *device_status, fp_stream_t stream) {
    Sizes s;
    fp_status st = describe(p, &s);
    if (st != FP_OK) return st;
    const WsLayout w = layout(p, s);
    // fp_select touches nothing from the split partial outputs on
    if (w.part_lse > kNoAllocScratchBytes) {
        fprintf(stderr,
                "libfp: fp_select_noalloc: this problem needs %lld bytes of scratch but the library's static "
                "scratch holds %lld; use fp_select with a caller-provided workspace\n",
                (long long)w.part_lse, (long long)kNoAllocScratchBytes);
        return FP_ERR_WORKSPACE;
    }
    if (!(alpha >= 0.f) || sink_blocks < 0 || window_blocks < 0 || csr_idx_capacity < 0) return FP_ERR_INVALID_ARG;
    if (!csr_cu) return FP_ERR_INVALID_ARG;
    if ((s.total_tokens > 0 && !q) ||
        (s.nblocks > 0 && (!k_pages || !v_pages || !kbar || !vbar || !kbar_op || !vbar_op)))
        return FP_ERR_INVALID_ARG;
    if (s.nseg > 0 && !csr_idx) return FP_ERR_INVALID_ARG;
    // tensors read through TMA start on 16-byte boundaries (as for fp_select)
    for (const void *t : {q, k_pages, v_pages, (const void *)kbar_op, (const void *)vbar_op})
        if (reinterpret_cast<uintptr_t>(t) & 15) return FP_ERR_INVALID_ARG;
    // the int32 / fp32 outputs on 4-byte ones
    for (const void *t : {(const void *)csr_cu, (const void *)csr_idx, (const void *)kbar, (const void *)vbar,
                          (const void *)device_status})
        if (reinterpret_cast<uintptr_t>(t) & 3) return FP_ERR_INVALID_ARG;
    char *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != FP_OK) return st;
    Ctx c;
    c.p = *p;
    c.s = s;
    c.ws = w;
    c.wsbase = scratch;
    c.stream = reinterpret_cast<cudaStream_t>(stream);
    // Only the status word must start at zero; every other region is fully
    // rewritten by the kernels before it is read.
    cudaError_t e = cudaMemsetAsync(c.status(), 0, 64 * 4, c.stream);
    if (e == cudaSuccess) e = launch_prep(c);
    if (e == cudaSuccess && s.nblocks > 0) e = launch_pool(c, k_pages, v_pages, kbar, vbar, kbar_op, vbar_op);
    if (e == cudaSuccess && s.nseg > 0) e = launch_score(c, q, kbar, kbar_op, alpha, sink_blocks, window_blocks);
    if (e == cudaSuccess) e = launch_csr(c, csr_cu, csr_idx, csr_idx_capacity);
    if (e == cudaSuccess && device_status)
        e = cudaMemcpyAsync(device_status, c.status(), sizeof(int32_t), cudaMemcpyDeviceToDevice, c.stream);
    if (e != cudaSuccess) {
        fprintf(stderr, "libfp: CUDA error: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    return FP_OK;
}
