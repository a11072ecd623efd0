// ssd_static.cu -- a forward entry point that allocates nothing, not even its workspace.
//
// Some callers cannot hand the library a workspace: a plugin inside a serving
// process or framework whose device memory is owned by the host application's
// pool, or a latency-critical loop where cudaMalloc (which can synchronise the
// device and can fail under memory pressure) is not allowed.  For them,
// ssd_varlen_forward_static runs the same plan + forward as ssd_varlen_plan and
// ssd_varlen_forward, but its workspace is a fixed array in device memory that
// belongs to the library (a file-scope __device__ array of
// SSD_STATIC_SCRATCH_BYTES bytes, held on each GPU that loads this code until
// the process exits).
//
// Rules of use (see include/ssd_varlen.h):
// * The first call on a device looks up the array's device address
//   (cudaGetSymbolAddress) with that device current; make that first call
//   before any stream capture on that device.
// * Every call shares the one array and it keeps the last call's contents:
//   calls whose work overlaps on the GPU (other streams, other host threads)
//   race on it; order them on one stream.  The metadata builder rewrites the
//   parts that must start from a known value (error word, counters) on every
//   call.
// * Problems whose workspace would exceed the array are rejected with
//   SSD_ERR_WORKSPACE before anything is launched.
#include <mutex>

#include "ssd_internal.cuh"

namespace ssd {
namespace {

__device__ __align__(256) unsigned char g_static_scratch[SSD_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
void *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of the scratch array on the current device (looked up once per device).
void *scratch_on_current_device() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_ptr[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_static_scratch) != cudaSuccess) return nullptr;
        g_scratch_ptr[dev] = ptr;
    }
    return g_scratch_ptr[dev];
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_varlen_forward_static(const ssd_dims *dims, const int32_t *cu_seqlens,
                                         const int32_t *num_computed, const ssd_inputs *in,
                                         const ssd_outputs *out, cudaStream_t stream, ssd_plan *plan_out) {
    if (!dims || !in || !out) return SSD_ERR_NULL;
    const size_t need = ssd_varlen_workspace_size(dims);
    if (need == 0) {
        ssd_plan probe;
        const int rc = ssd_varlen_plan(dims, cu_seqlens, num_computed, nullptr, 0, stream, &probe);
        return rc != SSD_OK ? rc : SSD_ERR_DIMS;  // reports the dims error without launching
    }
    if (need > (size_t)SSD_STATIC_SCRATCH_BYTES) return SSD_ERR_WORKSPACE;
    void *ws = ssd::scratch_on_current_device();
    if (!ws) return SSD_ERR_CUDA;
    ssd_plan plan;
    int rc = ssd_varlen_plan(dims, cu_seqlens, num_computed, ws, (size_t)SSD_STATIC_SCRATCH_BYTES, stream, &plan);
    if (rc != SSD_OK) return rc;
    rc = ssd_varlen_forward(&plan, in, out, stream);
    if (plan_out) *plan_out = plan;
    return rc;
}
