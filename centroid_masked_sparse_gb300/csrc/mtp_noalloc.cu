// mtp_masked_topk_tokens_noalloc: the sparse-argmax call for callers that
// cannot allocate device memory.
//
// Some callers are handed only their input and output buffers: a plugin or
// custom-operator interface of a host framework that passes tensors but no
// allocator, or a latency-critical path where cudaMalloc (which may
// synchronise the whole device) is not acceptable.  They cannot provide the
// workspace that mtp_masked_topk_tokens needs.  This entry point uses a
// scratch array that lives in the library's own device memory instead: a
// file-scope __device__ array of MTP_NOALLOC_SCRATCH_BYTES, which every GPU
// that loads the library holds until the process exits.
//
// In host code the array's name is only a host-side stand-in for the symbol,
// not a device address, so its device address is looked up once per device
// with cudaGetSymbolAddress (with that device current) and cached.  The call
// then runs the same kernels as mtp_masked_topk_tokens with that address as
// the workspace, whose first word is the device error word of the last call
// (mtp_noalloc_read_device_error reads it).  Nothing here allocates or frees
// memory.
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[MTP_NOALLOC_SCRATCH_BYTES];

std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_scratch on `dev` (current while it is looked up, on the
// first call for that device).
mtp_status scratch_address(int dev, void **addr)
{
    if (dev < 0 || dev >= kMaxDevices) return MTP_ERR_SHAPE;
    const mtp::DeviceScope scope(dev);
    if (!scope.ok) return MTP_ERR_CUDA;
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MTP_ERR_CUDA;
        g_noalloc_addr[dev] = p;
    }
    *addr = g_noalloc_addr[dev];
    return MTP_OK;
}

}  // namespace

extern "C" MTP_API mtp_status mtp_masked_topk_tokens_noalloc(const mtp_head_desc *desc,
                                                             const void *hidden, int32_t batch,
                                                             int32_t *out_tokens, float *out_max,
                                                             void *stream)
{
    // the same checks, in the same order, as the workspace entry point; only then the
    // size limit and the scratch address
    const mtp_status st = mtp::check_topk_call(desc, hidden, batch, out_tokens);
    if (st != MTP_OK || batch == 0) return st;
    const size_t need = mtp_workspace_bytes(desc, batch);
    if (need == 0) return MTP_ERR_SHAPE;
    if (need > (size_t)MTP_NOALLOC_SCRATCH_BYTES) return MTP_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const mtp_status sa = scratch_address(desc->device, &scratch);
    if (sa != MTP_OK) return sa;
    return mtp_masked_topk_tokens(desc, hidden, batch, out_tokens, out_max, scratch,
                                  (size_t)MTP_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" MTP_API mtp_status mtp_noalloc_read_device_error(int32_t device, uint32_t *host_word, void *stream)
{
    if (!host_word) return MTP_ERR_NULL;
    void *scratch = nullptr;
    const mtp_status st = scratch_address(device, &scratch);
    if (st != MTP_OK) return st;
    const mtp::DeviceScope scope(device);
    if (!scope.ok) return MTP_ERR_CUDA;
    return mtp_read_device_error(scratch, host_word, stream);
}
