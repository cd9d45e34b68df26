// common.cuh -- small device helpers shared by the libgdn kernels:
// mbarrier and bulk-copy (TMA) wrappers written as inline PTX for sm_103a,
// bounded waits, the device error word, and bf16 conversion.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

// Device error word values (the host maps them to gdn_status codes).
enum DevErr : int {
  kDevOk = 0,
  kDevTimeout = 1,     // a bounded mbarrier wait ran out
  kDevBadSeqlens = 2,  // cu_seqlens is not a valid offset table
  kDevOverlap = 3,     // a state_in pointer points into the slot buffer
  kDevGateRange = 4,   // a chunk's cumulative log-gate leaves [-80, 80] (chunked path)
};

// Where a bounded wait ran out: bits 8..15 of a timeout error word. The host
// names each site in the message of gdn_check_device_error.
enum WaitSite : int {
  kSiteRecTile = 11,      // recurrent kernel: token tile copies
  kSitePrepLoad = 21,     // chunk prep: K and Q tile copies
  kSitePrepG = 22,        // chunk prep: G product
  kSitePrepW = 23,        // chunk prep: W product
  kSiteScanX = 31,        // chunk scan, state warps: X product
  kSiteScanS = 32,        // chunk scan, state warps: state-update product
  kSiteScanO = 34,        // chunk scan, state warps: output product
  kSiteScanEmpty = 41,    // chunk scan, producer: a stage released by its products
  kSiteScanPad = 42,      // chunk scan, producer: copies of a partial last chunk
  kSiteScanReady = 43,    // chunk scan, producer: a tile of the chunk prep running beside it
  kSiteScanStage = 52,    // chunk scan, MMA issuer: a stage's copies
  kSiteScanS0 = 53,       // chunk scan, MMA issuer: the state operand
  kSiteScanD = 54,        // chunk scan, MMA issuer: the D tile
};

// Largest |cumulative log-gate| inside one chunk that the chunked kernels
// accept: their decay factors e^(+-gamma) are stored in bf16/fp32, whose
// range ends near e^88.
constexpr float kMaxChunkLogDecay = 80.f;

// Upper bound on polls of one mbarrier wait. A healthy wait completes in a
// few thousand polls; ~2^26 polls take well over a second.
constexpr uint32_t kMaxPolls = 1u << 26;

__device__ __forceinline__ void set_error(int *err, int code) {
  if (err) atomicCAS(err, 0, code);
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---- mbarrier ------------------------------------------------------------

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(count)
               : "memory");
}

// Makes barrier initialisation visible to the async proxy (TMA, tcgen05).
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar,
                                                      uint32_t bytes) {
  asm volatile(
      "mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(
          smem_u32(bar)),
      "r"(bytes)
      : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Waits for phase `parity` of `bar` to complete, polling at most max_polls
// times. Returns false (and sets the error word, with `site` in bits 8..15)
// if the wait ran out.
__device__ __forceinline__ bool mbar_wait_n(uint64_t *bar, uint32_t parity, int *err,
                                            int site, uint32_t max_polls) {
  for (uint32_t i = 0; i < max_polls; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  set_error(err, kDevTimeout | (site << 8));
  return false;
}

__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          int *err, int site = 0) {
  return mbar_wait_n(bar, parity, err, site, kMaxPolls);
}

// Orders this thread's generic-proxy shared-memory accesses before later
// async-proxy accesses (TMA copies and stores, tcgen05.mma operands).
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---- programmatic dependent launch ------------------------------------------
// Launch with programmatic stream serialisation allowed: the kernel may be
// scheduled once every block of the previous kernel in the stream has
// executed griddepcontrol.launch_dependents; it must execute
// griddepcontrol.wait before touching memory that kernel may write.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// ---- bulk copies (TMA, non-tensor form) ------------------------------------

// Global -> shared copy of `bytes` (multiple of 16, both addresses 16-byte
// aligned), completing on `bar` with complete_tx.
__device__ __forceinline__ void bulk_g2s(void *dst_smem, const void *src_gmem,
                                         uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes "
      "[%0], [%1], %2, [%3];" ::"r"(smem_u32(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// ---- global memory access --------------------------------------------------

__device__ __forceinline__ float4 ld_stream_f4(const float *p) {
  float4 r;
  asm volatile(
      "ld.global.nc.L1::no_allocate.v4.f32 {%0, %1, %2, %3}, [%4];"
      : "=f"(r.x), "=f"(r.y), "=f"(r.z), "=f"(r.w)
      : "l"(p));
  return r;
}

// Ordinary 16-byte load, issued where it stands (volatile, so that it is not
// moved behind later loads); page-locked host memory mapped into the
// device's address space is read this way too.
__device__ __forceinline__ uint4 ld_u4(const void *p) {
  uint4 r;
  asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ void st_f4(float *p, float4 v) {
  asm volatile("st.global.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(p), "f"(v.x),
               "f"(v.y), "f"(v.z), "f"(v.w)
               : "memory");
}

template <typename T>
__device__ __forceinline__ float to_f32(T x);
template <>
__device__ __forceinline__ float to_f32<float>(float x) {
  return x;
}
template <>
__device__ __forceinline__ float to_f32<__nv_bfloat16>(__nv_bfloat16 x) {
  return __bfloat162float(x);
}

}  // namespace gdn
