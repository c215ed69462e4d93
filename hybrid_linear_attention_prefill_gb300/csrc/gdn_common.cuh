// Shared device helpers for the chunked Gated DeltaNet prefill kernels (sm_103a).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

namespace gdn {

constexpr int kChunk = 64;  // tokens per chunk

// ---------------------------------------------------------------------------
// Workspace layout, per (chunk slot, value head): the UT-transform matrix Tm = (I + A)^-1
// and the decayed score product PT = P Tm, both 64 x 64 row-major, fp16 for the default
// state carry and bf16 for the wide-range one.
// ---------------------------------------------------------------------------
constexpr int kWsTileElems = kChunk * kChunk;           // 4096 16-bit elements
constexpr size_t kWsPerSlotHead = 2 * kWsTileElems * 2;  // bytes (Tm + PT)
// After the tiles, per (chunk slot, key head): the inverse L2 norms of the chunk's
// k rows then q rows (fp32, 64 + 64), written by the preparation kernel when q and k
// are normalised in-kernel.
constexpr size_t kWsNormPerSlotKHead = 2 * kChunk * 4;  // bytes
// After the norms, per (chunk slot, key head), for the fp16 state carry: the chunk's k rows
// then q rows as fp16 (normalised when q and k are normalised in-kernel), stored as the image
// of the shared-memory tile the state carry reads -- [dk/64 blocks of 16 KiB][128 rows][128 B],
// 128-byte swizzle, rows past the chunk's tokens zero -- so that one bulk copy restores it.
__host__ __device__ constexpr size_t kws_kq_bytes(int dk) { return (dk > 64 ? 2 : 1) * (size_t)16384; }
// Before the tiles (after 256 bytes of status words): the packed chunk table, B + 1 int32
// chunk offsets, then the B sequences in the order their state carries are dispatched
// (most chunks first), padded to 256 bytes.
inline size_t chunk_table_bytes(int B) { return (sizeof(int32_t) * (2 * (size_t)B + 1) + 255) / 256 * 256; }

struct SeqChunk {
  long long bos;  // first token of the sequence
  int len;        // tokens in the sequence
};

// Bounds of sequence b, clamped to [0, Ttot].
__device__ __forceinline__ SeqChunk seq_bounds(const int32_t* __restrict__ cu, int b, int T) {
  SeqChunk s;
  if (cu == nullptr) {
    s.bos = (long long)b * T;
    s.len = T;
  } else {
    int lo = cu[b], hi = cu[b + 1];
    lo = lo < 0 ? 0 : (lo > T ? T : lo);
    hi = hi < lo ? lo : (hi > T ? T : hi);
    s.bos = lo;
    s.len = hi - lo;
  }
  return s;
}

// ---------------------------------------------------------------------------
// bf16 helpers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);  // .x = lo (low 16 bits), .y = hi
  return *reinterpret_cast<uint32_t*>(&v);
}

// Split (a, b) into bf16 hi parts and bf16 residuals: a ~= hi.x + lo.x exactly to ~2^-17.
__device__ __forceinline__ void split_bf16(float a, float b, uint32_t& hi, uint32_t& lo) {
  __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  float2 hf = __bfloat1622float2(h);
  __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  hi = *reinterpret_cast<uint32_t*>(&h);
  lo = *reinterpret_cast<uint32_t*>(&l);
}

// ---------------------------------------------------------------------------
// mma.sync m16n8k16 bf16 -> fp32, and ldmatrix
// ---------------------------------------------------------------------------
__device__ __forceinline__ void mma_bf16(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
      "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
      : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void* p) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(smem_u32(p)));
}

// ---------------------------------------------------------------------------
// cp.async (16-byte and 4-byte, with zero fill when src_bytes == 0)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 16 : 0));
}

__device__ __forceinline__ void cp_async4(void* smem, const void* gmem, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;\n" ::"r"(smem_u32(smem)), "l"(gmem),
               "r"(valid ? 4 : 0));
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }

template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;\n" ::"n"(N));
}

// Raise a kernel's dynamic shared-memory limit once per device.  Doing it once keeps
// later calls free of runtime configuration calls, e.g. while a stream is being captured
// into a CUDA graph.  One flag set per kernel (the kernel is the template argument);
// the flags are atomic, so concurrent first calls from several host threads at worst
// both set the (same) attribute.
template <auto kernel>
inline cudaError_t set_smem_limit_once(int bytes) {
  static std::atomic<bool> done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire)) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
  return e;
}

}  // namespace gdn
