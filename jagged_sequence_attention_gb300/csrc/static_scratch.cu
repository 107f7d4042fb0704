// jfa_bwd_static_scratch: the backward pass with its scratch held by the library.
//
// jfa_bwd needs scratch: the softmax row terms [T_q, H], and (for fp32 inputs, and bf16
// inputs on the fused backward) an fp32 dQ accumulator [T_q, H, D] into which every
// key/value tile adds its share.
// Callers of jfa_bwd must pass that scratch in, which some cannot do.  Such callers include
// host code that owns no device allocator (the memory it works in was handed to it
// by another runtime), and programs whose device memory is all reserved by a pool
// set up at start, where a further cudaMalloc fails or breaks the pool's
// accounting.  For them this entry point keeps the scratch in one fixed-size
// device array that is part of the library image.  The array is created when the
// library's module loads on a GPU and stays until the process exits.
//
// Set-up: host code cannot use the array's name as a device address, because on the
// host that name is only a stand-in symbol.  The first call in each CUDA context
// (normally one per device: the device's primary context) therefore asks the runtime
// for the array's device address (cudaGetSymbolAddress, with that device current) and
// remembers it under the context's unique id; later calls in the same context reuse
// it.  A context created later -- after cudaDeviceReset, or a caller's own driver-API
// context -- has a new id and gets its own look-up, so no call ever hands a kernel an
// address that belongs to another context.  That first call may load the module on the
// device, so make it before any stream capture.
//
// The launches themselves are those of jfa_bwd, given the array as its workspace:
// the preprocess writes every row term before a later kernel reads one and clears
// the dQ accumulator, where there is one, on the stream before anything adds to it.
// So a call never depends on what an earlier call left in the array.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "jfa_internal.h"

// Scratch of every jfa_bwd_static_scratch call on a device (row terms, then for fp32
// inputs the dQ accumulator, each starting on a 256-byte boundary as in jfa_bwd's
// workspace).
static __device__ __align__(256) unsigned char jfa_static_bwd_scratch[JFA_STATIC_SCRATCH_BYTES];

namespace {

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Unique id of the calling thread's current context (ids are never reused within a
// process); false if there is none or the driver cannot say.
bool current_context_id(unsigned long long* id) {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return false;
    CUcontext ctx = nullptr;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx) return false;
    return get_id(ctx, id) == CUDA_SUCCESS;
}

// The array's address in each context seen so far, keyed by context id.
constexpr int kMaxContexts = 64;
std::mutex g_setup_mutex;
unsigned long long g_ctx_id[kMaxContexts] = {};
void* g_scratch_addr[kMaxContexts] = {};
int g_n_ctx = 0;

// Device address of the array in the current context; nullptr on failure.
void* scratch_address() {
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    unsigned long long id = 0;
    bool have_id = current_context_id(&id);
    if (have_id)
        for (int i = 0; i < g_n_ctx; ++i)
            if (g_ctx_id[i] == id) return g_scratch_addr[i];
    // First call in this context.  With no context current yet, this runtime call makes
    // the device's primary context current; its id is read afterwards.
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, jfa_static_bwd_scratch) != cudaSuccess || !ptr) return nullptr;
    if (!have_id) {
        have_id = current_context_id(&id);
        if (!have_id) return ptr;  // no id to key it by: look it up again next call
        for (int i = 0; i < g_n_ctx; ++i)
            if (g_ctx_id[i] == id) return g_scratch_addr[i];
    }
    // Remember it (with the table full, later contexts look it up on every call).
    if (g_n_ctx < kMaxContexts) {
        g_ctx_id[g_n_ctx] = id;
        g_scratch_addr[g_n_ctx] = ptr;
        ++g_n_ctx;
    }
    return ptr;
}

}  // namespace

extern "C" jfa_status jfa_bwd_static_scratch(jfa_plan plan, int32_t dtype, const void* Q, const void* K,
                                             const void* V, const void* O, int32_t o_dtype, const void* dO,
                                             const float* lse, int32_t bias_kind, const float* bias_table,
                                             float scale, void* dQ, void* dK, void* dV, void* stream) {
    if (!plan || (dtype != JFA_BF16 && dtype != JFA_F32)) return JFA_ERR_INVALID_ARG;
    if (jfa_bwd_workspace_size(plan, dtype) > JFA_STATIC_SCRATCH_BYTES) return JFA_ERR_SCRATCH_LIMIT;
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return JFA_ERR_NO_DEVICE;
    if (dev != plan->device) return JFA_ERR_PLAN_MISMATCH;
    void* scratch = scratch_address();
    if (!scratch) return JFA_ERR_CUDA;
    return jfa_bwd(plan, dtype, Q, K, V, O, o_dtype, dO, lse, bias_kind, bias_table, scale, dQ, dK, dV, scratch,
                   JFA_STATIC_SCRATCH_BYTES, stream);
}
