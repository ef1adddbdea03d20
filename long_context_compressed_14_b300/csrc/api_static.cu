// api_static.cu -- csa_decode for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: a host application whose device memory belongs
// to another framework's allocator that gives out no scratch buffers, a real-time serving loop
// that must not call cudaMalloc (it can synchronise the device and take unbounded time), or a
// caller held to a fixed device-memory budget. csa_decode needs scratch (indexer scores and the
// selected indices); this entry point takes it from one fixed array compiled into the library
// instead of from the caller.
//
// The array is file-scope device memory of CSA_STATIC_SCRATCH_BYTES: every GPU that loads the
// library holds it until the process exits. In host code its name is only a host-side
// stand-in, so its device address is looked up with cudaGetSymbolAddress -- once per device,
// on the first call made with that device current -- and that address is what the kernels
// receive. All calls on a device share the array: calls that overlap on the GPU (different
// streams without ordering between them) race on it. Nothing in it needs to start at zero:
// every decode step writes the scores and indices before it reads them.
#include <mutex>

#include "common.cuh"

namespace {

__device__ __align__(256) unsigned char g_decode_scratch[CSA_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of the array on the current device; set up once per device.
int scratch_address(void **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CSA_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CSA_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_addr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_decode_scratch) != cudaSuccess || !ptr) return CSA_ERR_CUDA;
        g_scratch_addr[dev] = ptr;
    }
    *out = g_scratch_addr[dev];
    return CSA_OK;
}

}  // namespace

extern "C" int csa_decode_static_scratch(const csa_params *p, const void *q, const int32_t *ctx_len,
                                         const csa_entries *C, const csa_index_rows *qI,
                                         const csa_index_rows *KI, const float *w, const void *swa_ring,
                                         const float *sink, const float *rope_tab, int32_t *topk_out,
                                         void *out, float *lse_out, csa_stream_t stream) {
    const int s = csa_check_params(p, CSA_OP_CSA_DECODE);
    if (s != CSA_OK) return s;
    // the layer's scratch must fit the fixed array: refuse larger layers before any launch
    if (csa_workspace_bytes(p, CSA_OP_CSA_DECODE) > (size_t)CSA_STATIC_SCRATCH_BYTES) return CSA_ERR_WORKSPACE;
    void *scratch = nullptr;
    const int a = scratch_address(&scratch);
    if (a != CSA_OK) return a;
    return csa_decode(p, q, ctx_len, C, qI, KI, w, swa_ring, sink, rope_tab, topk_out, out, lse_out, scratch,
                      (size_t)CSA_STATIC_SCRATCH_BYTES, stream);
}
