// validate.cu -- device check of the index values a decode step will use.
//
// The pages gate every span before the GPU touches it (mainarch, kernel-ABI
// layer: every buffer checked before dispatch; Loom Kernels, "What Loom
// owns": invalid-input behaviour is part of each operator's contract). The
// hot kernels already skip and flag bad indices; this kernel lets a caller
// check a whole batch's metadata up front, including duplicate slots, which
// the write kernel cannot see.
//
// Threads [0, 32*B) work one warp per sequence (its seq_len, then the
// block-table entries it needs, lanes striding over pages); threads
// [32*B, 32*B + T) check one slot_mapping entry each and, given a bitmap of
// one bit per cache slot, set the slot's bit with atomicOr: a bit that was
// already set marks a duplicate.
#include <mutex>

#include "pkv_internal.h"
#include "pkv_ptx.cuh"

namespace pkv {
namespace {

__global__ void __launch_bounds__(256) validate_kernel(const ValidateArgs a) {
    const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    const int64_t nseq = static_cast<int64_t>(a.B) * 32;
    if (idx < nseq) {
        const int b = static_cast<int>(idx >> 5);
        const int lane = static_cast<int>(idx & 31);
        int L = a.seq_lens[b * a.sl_s0];
        const int cap = a.max_pages * kPageSize;
        if (L < 0 || L > cap) {
            if (lane == 0) flag_error(a.err, PKV_FLAG_SEQ_LEN_RANGE);
            L = L < 0 ? 0 : cap;
        }
        const int npages = (L + kPageSize - 1) / kPageSize;
        bool bad = false;
        for (int p = lane; p < npages; p += 32) {
            const int32_t pid = a.block_tables[b * a.bt_s0 + p * a.bt_s1];
            bad |= (pid < 0 || pid >= a.num_pages);
        }
        if (bad) flag_error(a.err, PKV_FLAG_PAGE_RANGE);
        return;
    }
    const int64_t t = idx - nseq;
    if (a.slots == nullptr || t >= a.T) return;
    const int32_t slot = a.slots[t * a.sm_s0];
    if (slot < 0) return;
    if (slot >= a.num_pages * kPageSize) {
        flag_error(a.err, PKV_FLAG_SLOT_RANGE);
        return;
    }
    if (a.bitmap) {
        const uint32_t bit = 1u << (slot & 31);
        const uint32_t old = atomicOr(a.bitmap + (slot >> 5), bit);
        if (old & bit) flag_error(a.err, PKV_FLAG_DUPLICATE_SLOT);
    }
}

// Bitmap for pkv_validate_indices_static: a fixed device array so that the
// entry point needs no allocation. Host code must not pass the symbol itself
// to a kernel (on the host it names a host-side stand-in, not device
// memory): static_slot_bitmap() looks up its device address.
static __device__ __align__(256) uint32_t g_static_slot_bitmap[PKV_STATIC_VALIDATE_MAX_SLOTS / 32];

}  // namespace

// Device address of this device's copy of the static bitmap, looked up with
// that device current. A successful lookup is kept and reused; a failed one
// is not (the next call on that device tries again), so a lookup that fails
// for a passing reason -- made during a stream capture, or before the device
// was ready -- does not disable the entry point for the rest of the process.
cudaError_t static_slot_bitmap(uint32_t** ptr, int64_t* words) {
    constexpr int kMaxDevices = 64;
    static uint32_t* addr[kMaxDevices] = {};
    static std::mutex lock[kMaxDevices];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    {
        std::lock_guard<std::mutex> guard(lock[dev]);
        if (addr[dev] == nullptr) {
            void* p = nullptr;
            e = cudaGetSymbolAddress(&p, g_static_slot_bitmap);
            if (e != cudaSuccess) {
                (void)cudaGetLastError();  // leave no sticky error behind for the caller's next launch
                return e;
            }
            addr[dev] = static_cast<uint32_t*>(p);
        }
        *ptr = addr[dev];
    }
    *words = PKV_STATIC_VALIDATE_MAX_SLOTS / 32;
    return cudaSuccess;
}

cudaError_t launch_validate(const ValidateArgs& a, cudaStream_t s) {
    if (a.bitmap) {
        cudaError_t e = cudaMemsetAsync(a.bitmap, 0, static_cast<size_t>(a.bitmap_words) * 4, s);
        if (e != cudaSuccess) return e;
    }
    const int64_t total = static_cast<int64_t>(a.B) * 32 + (a.slots ? a.T : 0);
    if (total == 0) return cudaSuccess;
    const int64_t blocks = (total + 255) / 256;
    if (blocks > 0x7FFFFFFF) return cudaErrorInvalidConfiguration;
    validate_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(a);
    return cudaGetLastError();
}

}  // namespace pkv
