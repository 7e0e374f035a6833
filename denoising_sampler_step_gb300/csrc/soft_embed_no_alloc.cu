// dg_soft_embed_no_alloc: the soft-embed product for callers that cannot allocate
// device memory.
//
// dg_soft_embed asks the caller for a workspace that holds the split-K partial
// tiles.  Some callers have no way to provide one: code that runs inside another
// framework's memory pool or under a fixed memory budget, plugins that are handed
// only the input and output buffers, or a process that must not allocate device
// memory once it is serving.  This entry point takes the same inputs and outputs
// and keeps its partial tiles in a fixed array compiled into the library instead.
//
// The array is kStaticScratchBytes large and every GPU that loads the library holds
// it until the process exits.  A shape whose partial tiles do not fit, even with a
// single split, is rejected with DG_ERR_UNSUPPORTED.  The array is shared by all
// calls on a device and keeps the last call's contents: every call rewrites each
// partial tile it later reads, so nothing has to be cleared, but two calls whose
// kernels overlap on the GPU (different streams, no ordering between them) race on
// it.  The first call on each device looks up the array's device address (with that
// device current), and so does the first call after the device's context was created
// anew (a device reset reloads the library's device code at another address); make those
// calls before any stream capture.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "dg_common.cuh"
#include "dg_internal.h"

namespace dg {

namespace {

constexpr size_t kStaticScratchBytes = size_t(16) << 20;  // 16 MiB per device

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

constexpr int kMaxScratchDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxScratchDevices] = {};
unsigned long long g_scratch_ctx[kMaxScratchDevices] = {};  // context the address belongs to

// Unique id of the calling thread's current CUDA context (0 when there is none or the driver
// cannot tell): a context created anew after a reset gets another id.
unsigned long long current_context_id() {
    typedef CUresult (*GetCurrent)(CUcontext *);
    typedef CUresult (*GetId)(CUcontext, unsigned long long *);
    static GetCurrent get_current = nullptr;
    static GetId get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *a = nullptr, *b = nullptr;
        cudaDriverEntryPointQueryResult q1, q2;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &a, 12000, cudaEnableDefault, &q1) == cudaSuccess &&
            q1 == cudaDriverEntryPointSuccess &&
            cudaGetDriverEntryPointByVersion("cuCtxGetId", &b, 12000, cudaEnableDefault, &q2) == cudaSuccess &&
            q2 == cudaDriverEntryPointSuccess) {
            get_current = reinterpret_cast<GetCurrent>(a);
            get_id = reinterpret_cast<GetId>(b);
        }
    });
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (!get_current || get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of g_static_scratch on the current device: looked up once per device and
// again whenever the device's context is not the one the address was taken in (without a
// context id it is looked up on every call).
dg_status scratch_address(void **out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e, "soft embed (no alloc): no current device");
    if (dev < 0 || dev >= kMaxScratchDevices) return fail(DG_ERR_UNSUPPORTED, "soft embed (no alloc): device %d", dev);
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    const unsigned long long ctx = current_context_id();
    if (!g_scratch_ptr[dev] || ctx == 0 || g_scratch_ctx[dev] != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_static_scratch);
        if (e != cudaSuccess) return cuda_fail(e, "soft embed (no alloc): scratch address lookup");
        g_scratch_ptr[dev] = p;
        g_scratch_ctx[dev] = current_context_id();  // the lookup may have made the context current
    }
    *out = g_scratch_ptr[dev];
    return DG_OK;
}

}  // namespace

}  // namespace dg

using namespace dg;

extern "C" dg_status dg_soft_embed_no_alloc(const float *logits, int64_t ldl, const float *lse, int64_t R,
                                            int64_t vocab_start, int64_t vocab_end, const uint16_t *W_shard,
                                            int64_t rows_pad, int64_t ldw, int64_t d, float gamma, float *out,
                                            int64_t ldo, dg_stream_t stream) {
    t_last_error[0] = 0;
    dg_status st = check_embed_args(logits, ldl, lse, R, vocab_start, vocab_end, W_shard, rows_pad, ldw, d, out, ldo);
    if (st != DG_OK) return st;
    if (R == 0) return DG_OK;
    cudaStream_t s = (cudaStream_t)stream;
    if (vocab_end == vocab_start) {
        cudaError_t e = launch_fill_zero(out, R, d, ldo, s);
        return e == cudaSuccess ? DG_OK : cuda_fail(e, "soft embed (no alloc, empty slice)");
    }
    const int sms = device_sm_count();
    if (sms <= 0) return fail(DG_ERR_CUDA, "soft embed (no alloc): no CUDA device");
    SoftEmbedPlan plan;
    if (!plan_soft_embed(R, vocab_start, vocab_end, d, sms, &plan))
        return fail(DG_ERR_INVALID_ARG, "soft embed (no alloc): no plan for shape");
    // fewer vocabulary splits until the partial tiles fit the fixed scratch array
    const size_t one_split = soft_embed_workspace_bytes(plan, 1);
    if (one_split > kStaticScratchBytes)
        return fail(DG_ERR_UNSUPPORTED,
                    "soft embed (no alloc): %lld rows x %lld columns need %zu bytes of partial tiles, above the "
                    "%zu-byte fixed scratch; use dg_soft_embed with a workspace",
                    (long long)R, (long long)d, one_split, kStaticScratchBytes);
    const size_t fit = kStaticScratchBytes / one_split;
    if ((size_t)plan.splits > fit) plan.splits = (int)fit;
    plan.workspace_bytes = soft_embed_workspace_bytes(plan, plan.splits);
    void *scratch = nullptr;
    st = scratch_address(&scratch);
    if (st != DG_OK) return st;
    const char *msg = "soft embed (no alloc)";
    const EmbedTable tab{kTableBf16, W_shard, ldw, nullptr};
    cudaError_t e = launch_soft_embed(logits, ldl, lse, R, vocab_start, vocab_end, tab, d, gamma, out, ldo, scratch,
                                      plan, s, &msg);
    return e == cudaSuccess ? DG_OK : cuda_fail(e, msg);
}
