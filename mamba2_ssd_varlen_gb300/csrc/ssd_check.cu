// ssd_check.cu -- the slot-aliasing check for debug runs: no pool slot written
// by a call (final slots, block-table entries) may be read by it (initial
// slots) or written twice.  The forward, the decode step and the gated delta
// rule assume this and do not test it per call ("Automatic prefix caching for
// GDN hybrid models (mamba_cache_mode=all) with MTP speculative decoding",
// Purpose: dual read/write state anchors; the scatter listing writes one block
// slot per boundary).
#include "ssd_internal.cuh"

namespace ssd {
namespace {

constexpr int kCheckThreads = 256;

// Write slot number w of the call: final_slots[0..R), then the block table row by row.
__device__ __forceinline__ int write_slot(const int32_t *fin, const int32_t *bt, int R, int W, int64_t w) {
    if (w < R) return fin ? fin[w] : -1;
    return bt ? bt[w - R] : -1;
}

// One thread per write slot: compared with every read slot and every later write slot.
__global__ void check_slots_kernel(const int32_t *init, const int32_t *fin, const int32_t *bt, int R, int W,
                                   int32_t *err) {
    const int64_t nw = (int64_t)R + (int64_t)R * W;
    for (int64_t w = blockIdx.x * (int64_t)kCheckThreads + threadIdx.x; w < nw;
         w += (int64_t)gridDim.x * kCheckThreads) {
        const int s = write_slot(fin, bt, R, W, w);
        if (s < 0) continue;
        bool bad = false;
        if (init)
            for (int i = 0; i < R && !bad; ++i) bad = init[i] == s;
        for (int64_t v = w + 1; v < nw && !bad; ++v) bad = write_slot(fin, bt, R, W, v) == s;
        if (bad) atomicOr(err, SSD_DEVERR_ALIAS);
    }
}

}  // namespace
}  // namespace ssd

extern "C" int ssd_varlen_check_slots(const ssd_dims *dims, const int32_t *init_slots, const int32_t *final_slots,
                                      const int32_t *block_table, int32_t *device_err, cudaStream_t stream) {
    if (!dims || !device_err) return SSD_ERR_NULL;
    if (dims->R < 1 || dims->block_table_width < 0) return SSD_ERR_DIMS;
    const int W = block_table ? dims->block_table_width : 0;
    const int64_t nw = (int64_t)dims->R + (int64_t)dims->R * W;
    const int64_t blocks = (nw + ssd::kCheckThreads - 1) / ssd::kCheckThreads;
    ssd::check_slots_kernel<<<(unsigned)(blocks < 4096 ? blocks : 4096), ssd::kCheckThreads, 0, stream>>>(
        init_slots, final_slots, block_table, dims->R, W, device_err);
    return cudaGetLastError() == cudaSuccess ? SSD_OK : SSD_ERR_CUDA;
}
