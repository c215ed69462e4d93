// gdn_prefill_static: the prefill with its scratch in a fixed, file-scope device
// array, for callers that cannot allocate device memory.
//
// Who needs this.  gdn_prefill grows a library-owned workspace with cudaMalloc
// the first time a larger problem arrives.  Some callers cannot allow that: a
// plugin inside an inference engine that owns all device memory and gives its
// plugins none, code that runs with a fixed memory budget decided at start-up,
// or a caller that must not trigger the implicit device synchronisation that
// cudaMalloc/cudaFree bring.  This entry point takes only the caller's inputs
// and outputs and never allocates: its scratch (the chunk table and the per-chunk
// Tm / PT tiles, the fp16 k / q images) lives in `g_static_scratch` below, which every GPU that loads
// the library holds until the process exits.
//
// Limits and sharing.  The array holds GDN_STATIC_SCRATCH_BYTES; a call whose
// scratch (gdn_workspace_bytes for its sizes) does not fit returns
// GDN_ERR_SCRATCH before launching anything.  All calls on a device share the
// one array and it keeps the last call's contents; nothing in it has to start at
// zero (each call writes every entry it later reads), but two calls whose work
// overlaps on the GPU (different streams, or different host threads without
// ordering) race on it and must be serialised by the caller.
//
// Set-up.  The device address of the array is looked up once per device, with
// that device current, by the first call made on it (cudaGetSymbolAddress).
// Make that first call before capturing a stream into a CUDA graph.
//
// Status.  The kernels' status bits (a bounded wait that ran out, a malformed
// cu_seqlens) go to the array's first word; gdn_device_status reads and clears it
// together with the workspace's.
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"
#include "gdn_internal.h"
#include <climits>

namespace gdn {
template <int DK>
cudaError_t launch_prep(const void*, const void*, const float*, const float*, const int32_t*, const int32_t*,
                        void*, float*, void*, int, int*, int, int, int, int, int, int, int, int, int, int, int, int,
                        cudaStream_t);
cudaError_t launch_chunk_table(const int32_t*, int, int, int32_t*, int32_t*, int*, cudaStream_t);
cudaError_t launch_wait_timeout_probe(int max_polls, int* status, cudaStream_t st);
template <int DK>
cudaError_t launch_chain_f16(const void*, const float*, const float*, const int32_t*, const int32_t*,
                             const int32_t*, const void*, const void*, const float*, void*, float*, int*, int, int,
                             int, int, int, int, long long, int, int, int, int, int, int, cudaStream_t);
}  // namespace gdn

namespace {

static __device__ __align__(256) unsigned char g_static_scratch[GDN_STATIC_SCRATCH_BYTES];

constexpr int kMaxDev = 64;
std::mutex g_static_mu;
void* g_static_ptr[kMaxDev] = {};
size_t round256(size_t x) { return (x + 255) / 256 * 256; }

// The array's device address on the current device, looked up on first use.
cudaError_t static_base(int dev, void** base) {
  std::lock_guard<std::mutex> lock(g_static_mu);
  if (g_static_ptr[dev] == nullptr) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    if (p == nullptr) return cudaErrorInvalidSymbol;
    g_static_ptr[dev] = p;
  }
  *base = g_static_ptr[dev];
  return cudaSuccess;
}

}  // namespace

namespace gdn {
void* static_scratch_address(int dev) {
  if (dev < 0 || dev >= kMaxDev) return nullptr;
  std::lock_guard<std::mutex> lock(g_static_mu);
  return g_static_ptr[dev];
}
}  // namespace gdn

extern "C" int gdn_prefill_static(const void* q, const void* k, const void* v, const float* g,
                                  const float* beta, const int32_t* cu_seqlens, const float* init_state,
                                  void* out, float* final_state, int B, int T, int Hk, int Hv, int dk, int dv,
                                  void* stream) {
  gdn::clear_cuda_error();
  const bool dims_ok = (dk == 32 || dk == 64 || dk == 128) && (dv == 32 || dv == 64 || dv == 128);
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0 || !dims_ok || Hv > 65535) return GDN_ERR_ARG;
  if ((long long)B * (dv / 32) > 0x7fffffffLL) return GDN_ERR_ARG;
  if (B == 0) return GDN_OK;
  const int packed = cu_seqlens != nullptr;
  const long long ntok = packed ? (long long)T : (long long)B * T;
  if (ntok > 0x7fffffffLL) return GDN_ERR_ARG;
  if (ntok > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, init_state, out, final_state};
  for (const void* p : ptrs)
    if (p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) != 0) return GDN_ERR_ALIGN;
  if (ntok == 0 && final_state == nullptr) return GDN_OK;

  // scratch layout: [256 B status words][chunk table and dispatch order][Tm/PT tiles]
  //                 [inverse q/k norms per (slot, key head)][fp16 [K; Q] images per (slot, key head)]
  const long long nslots = packed ? (long long)(T + gdn::kChunk - 1) / gdn::kChunk + B
                                  : (long long)B * ((T + gdn::kChunk - 1) / gdn::kChunk);
  const size_t table = gdn::chunk_table_bytes(B);
  const size_t need = 256 + table + (size_t)nslots * Hv * gdn::kWsPerSlotHead +
                      (size_t)nslots * Hk * gdn::kWsNormPerSlotKHead + (size_t)nslots * Hk * gdn::kws_kq_bytes(dk);
  if (need > (size_t)GDN_STATIC_SCRATCH_BYTES || nslots > 0x7fffffffLL) return GDN_ERR_SCRATCH;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDev) return GDN_ERR_ARG;
  void* base = nullptr;
  if ((e = static_base(dev, &base)) != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);

  cudaStream_t st = static_cast<cudaStream_t>(stream);
  int* err = static_cast<int*>(base);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(base) + 256);
  int32_t* order = packed ? chunk_off + B + 1 : nullptr;  // packed: state carries longest first
  void* tiles = static_cast<unsigned char*>(base) + 256 + table;
  float* ws_rn = reinterpret_cast<float*>(static_cast<unsigned char*>(tiles) + (size_t)nslots * Hv * gdn::kWsPerSlotHead);
  void* ws_kq = reinterpret_cast<unsigned char*>(ws_rn) + (size_t)nslots * Hk * gdn::kWsNormPerSlotKHead;
  const int nc_dense = (T + gdn::kChunk - 1) / gdn::kChunk;
  if (packed) {
    e = gdn::launch_chunk_table(cu_seqlens, B, T, chunk_off, order, err, st);
    if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  // the gdn_set_phase_events hook: around the preparation and state-carry kernels
  cudaEvent_t ev[3];
  gdn::take_phase_events(ev);
  if (ev[0] != nullptr && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  if (nslots > 0) {
    switch (dk) {
      case 32: e = gdn::launch_prep<32>(q, k, g, beta, cu_seqlens, chunk_off, tiles, ws_rn, ws_kq, 1, err, B, T, Hk, Hv, (int)nslots, nc_dense, 0, 0, Hk, 0, nc_dense, 1, st); break;
      case 64: e = gdn::launch_prep<64>(q, k, g, beta, cu_seqlens, chunk_off, tiles, ws_rn, ws_kq, 1, err, B, T, Hk, Hv, (int)nslots, nc_dense, 0, 0, Hk, 0, nc_dense, 1, st); break;
      default: e = gdn::launch_prep<128>(q, k, g, beta, cu_seqlens, chunk_off, tiles, ws_rn, ws_kq, 1, err, B, T, Hk, Hv, (int)nslots, nc_dense, 0, 0, Hk, 0, nc_dense, 1, st); break;
    }
    if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  if (ev[1] != nullptr && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  switch (dk) {
    case 32: e = gdn::launch_chain_f16<32>(v, g, beta, cu_seqlens, chunk_off, order, tiles, ws_kq, init_state, out, final_state, err, B, T, Hk, Hv, dv, nc_dense, nslots, 0, Hv, 0, INT_MAX, 0, 1, st); break;
    case 64: e = gdn::launch_chain_f16<64>(v, g, beta, cu_seqlens, chunk_off, order, tiles, ws_kq, init_state, out, final_state, err, B, T, Hk, Hv, dv, nc_dense, nslots, 0, Hv, 0, INT_MAX, 0, 1, st); break;
    default: e = gdn::launch_chain_f16<128>(v, g, beta, cu_seqlens, chunk_off, order, tiles, ws_kq, init_state, out, final_state, err, B, T, Hk, Hv, dv, nc_dense, nslots, 0, Hv, 0, INT_MAX, 0, 1, st); break;
  }
  if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  if (ev[2] != nullptr && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

// The bounded-wait self-test with the static array's status word as its target: the bit
// it records is then read back by gdn_device_status, as a timed-out wait inside a
// gdn_prefill_static call would be.  Synchronous; allocates nothing.
extern "C" int gdn_selftest_static_wait_timeout(int max_polls) {
  gdn::clear_cuda_error();
  if (max_polls < 1) return GDN_ERR_ARG;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDev) return GDN_ERR_ARG;
  void* base = nullptr;
  if ((e = static_base(dev, &base)) != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  e = gdn::launch_wait_timeout_probe(max_polls, static_cast<int*>(base), nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return gdn::set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}
