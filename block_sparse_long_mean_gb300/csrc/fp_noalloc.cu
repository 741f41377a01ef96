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
#include <utility>

#include "fp_internal.cuh"

namespace fp {
namespace {

constexpr int64_t kNoAllocScratchBytes = int64_t(16) << 20;
constexpr int kMaxDevices = 64;

// The scratch itself. Host code may not use this name as a device address
// (on the host it only stands for the symbol); it asks the runtime for the
// address with cudaGetSymbolAddress instead.
static __device__ __align__(256) char g_noalloc_scratch[kNoAllocScratchBytes];

// The array's address belongs to one CUDA context: a device reset, or a
// different context made current on the same device, loads the library's
// device code again at another address. Addresses are therefore cached per
// context, keyed by the context's unique id (cuCtxGetId: never reused within
// the process, unlike a context handle).
struct ScratchEntry {
    unsigned long long ctx_id;
    char *ptr;
};
std::mutex g_mu;
ScratchEntry g_scratch[kMaxDevices] = {};
int g_scratch_n = 0, g_scratch_next = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);
using CtxGetIdFn = CUresult (*)(CUcontext, unsigned long long *);

// The unique id of the current context; false if the driver cannot say.
bool current_context_id(unsigned long long *id) {
    static const std::pair<CtxGetCurrentFn, CtxGetIdFn> fns = [] {
        void *cur = nullptr, *gid = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &cur, 12000, cudaEnableDefault, &q1) !=
                cudaSuccess || q1 != cudaDriverEntryPointSuccess)
            cur = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &gid, 12000, cudaEnableDefault, &q2) != cudaSuccess ||
            q2 != cudaDriverEntryPointSuccess)
            gid = nullptr;
        return std::make_pair(reinterpret_cast<CtxGetCurrentFn>(cur), reinterpret_cast<CtxGetIdFn>(gid));
    }();
    if (!fns.first || !fns.second) return false;
    CUcontext ctx = nullptr;
    if (fns.first(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return fns.second(ctx, id) == CUDA_SUCCESS;
}

// Device address of the scratch in the current context. The first call in
// each context (so the first on each device, and the first after a device
// reset) looks it up with cudaGetSymbolAddress; later calls take it from the
// cache. Without a context id the lookup is done on every call.
fp_status scratch_address(char **out) {
    // before the runtime's first call on a thread no context may be current yet: then the lookup below
    // makes the device's primary context current, and the next call finds it in the cache
    unsigned long long id = 0;
    const bool have_id = current_context_id(&id);
    std::lock_guard<std::mutex> lock(g_mu);
    if (have_id)
        for (int i = 0; i < g_scratch_n; ++i)
            if (g_scratch[i].ctx_id == id) {
                *out = g_scratch[i].ptr;
                return FP_OK;
            }
    void *ptr = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (e != cudaSuccess || !ptr) {
        fprintf(stderr, "libfp: cudaGetSymbolAddress of the static scratch failed: %s\n", cudaGetErrorString(e));
        return FP_ERR_CUDA;
    }
    if (have_id) {
        // oldest entry out when the table is full
        const int slot = g_scratch_n < kMaxDevices ? g_scratch_n++ : (g_scratch_next++ % kMaxDevices);
        g_scratch[slot] = ScratchEntry{id, static_cast<char *>(ptr)};
    }
    *out = static_cast<char *>(ptr);
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
