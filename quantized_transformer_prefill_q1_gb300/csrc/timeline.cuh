// timeline.cuh — optional per-CTA kernel timeline (pf_timeline_set in pf.h): the CUDA
// analogue of the GPU start / end stamps per command buffer of oxibonsai-kernels
// metal_full_layer.rs (OXIBONSAI_PROFILE_GPU), kept per CTA. Every kernel opens with
// PF_TIMELINE(id); while a buffer is set, the CTA's thread 0 appends
// {start ns, end ns, id << 48 | SM << 32 | linear CTA index, 0} when it leaves the kernel.
#pragma once
#include <cstdint>

namespace pf {
namespace tl {

// This translation unit's copy of the buffer address ([0] records appended, [1] capacity,
// records of 4 words from [4]); set by timeline_set_<unit> in the same file.
static __device__ unsigned long long* g_buf = nullptr;

struct Guard {
  unsigned long long t0;
  int id;
  __device__ __forceinline__ explicit Guard(int kernel_id) : t0(0), id(kernel_id) {
    if (threadIdx.x == 0 && threadIdx.y == 0 && threadIdx.z == 0)
      asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t0));
  }
  __device__ __forceinline__ ~Guard() {
    if (threadIdx.x != 0 || threadIdx.y != 0 || threadIdx.z != 0) return;
    unsigned long long* b = g_buf;
    if (b == nullptr) return;
    unsigned long long t1;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t1));
    unsigned smid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    const unsigned long long i = atomicAdd(b, 1ull);
    if (i >= b[1]) return;
    unsigned long long* r = b + 4 + 4 * i;
    const unsigned long long cta =
        blockIdx.x + static_cast<unsigned long long>(gridDim.x) * (blockIdx.y + static_cast<unsigned long long>(gridDim.y) * blockIdx.z);
    r[0] = t0;
    r[1] = t1;
    r[2] = (static_cast<unsigned long long>(id) << 48) | (static_cast<unsigned long long>(smid) << 32) |
           (cta & 0xffffffffull);
    r[3] = 0;
  }
};

}  // namespace tl
}  // namespace pf

#define PF_TIMELINE(id) ::pf::tl::Guard pf_timeline_guard_(id)
// Defines the host-side setter of this translation unit's buffer address.
#define PF_TIMELINE_SETTER(unit)                                                        \
  namespace pf {                                                                        \
  cudaError_t timeline_set_##unit(unsigned long long* buf) {                            \
    return cudaMemcpyToSymbol(tl::g_buf, &buf, sizeof(buf));                            \
  }                                                                                     \
  }
