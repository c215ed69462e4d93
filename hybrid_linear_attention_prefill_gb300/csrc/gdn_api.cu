// C ABI of the chunked Gated DeltaNet prefill library: argument checks, the
// per-device workspace, and the launch sequence
//   [packed only] chunk table  ->  chunk preparation  ->  chunk-sequential state carry.
// The interface style -- a versioned C ABI, scratch owned by the library and
// only ever grown, oversize or malformed requests refused before any work --
// follows the pages' native CUDA library ("Cua-S1 4B 0.2 native text worker",
// CUDA Graph paragraph; "Open-Jev-27B-v1.1 native text worker", "Build and
// serve" and "Prepare the checkpoint").
#include <mutex>

#include "../../include/gdn.h"
#include "gdn_common.cuh"

namespace gdn {
template <int DK>
cudaError_t launch_prep(const void*, const void*, const float*, const float*, const int32_t*, const int32_t*,
                        void*, int*, int, int, int, int, int, int, int, cudaStream_t);
cudaError_t launch_chunk_table(const int32_t*, int, int, int32_t*, cudaStream_t);
template <int DK>
cudaError_t launch_chain_tc(const void*, const void*, const void*, const float*, const float*, const int32_t*,
                            const int32_t*, const void*, const float*, void*, float*, int*, int, int, int, int, int,
                            int, long long, int, cudaStream_t);
cudaError_t launch_wait_timeout_probe(int max_polls, int* status, cudaStream_t st);
template <int DK>
cudaError_t launch_decode(const void*, const void*, const void*, const float*, const float*, float*, void*, int,
                          int, int, int, cudaStream_t);
}  // namespace gdn

namespace {

constexpr int kMaxDevices = 64;

struct DevBuffers {
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* stage = nullptr;  // device staging for gdn_prefill_host
  size_t stage_bytes = 0;
};

std::mutex g_mu;
DevBuffers g_dev[kMaxDevices];
thread_local int t_last_cuda_error = 0;
thread_local cudaEvent_t t_phase_ev[3] = {nullptr, nullptr, nullptr};

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool dim_ok(int d) { return d == 32 || d == 64 || d == 128; }

int check_sizes(int B, int T, int Hk, int Hv, int dk, int dv) {
  if (B < 0 || T < 0 || Hk <= 0 || Hv <= 0 || Hv % Hk != 0) return GDN_ERR_ARG;
  if (!dim_ok(dk) || !dim_ok(dv)) return GDN_ERR_ARG;
  if (Hv > 65535) return GDN_ERR_ARG;                 // grid.y
  if ((long long)B * (dv / 32) > 0x7fffffffLL) return GDN_ERR_ARG;  // grid.x
  return GDN_OK;
}

// Chunk slots: exact for equal-length sequences, an upper bound when packed.
long long num_slots(int B, int T, int packed) {
  if (!packed) return (long long)B * ((T + gdn::kChunk - 1) / gdn::kChunk);
  return (long long)(T + gdn::kChunk - 1) / gdn::kChunk + B;
}

// Workspace: [256 B status words][chunk table, B + 1 int32, padded to 256 B][Tm/PT tiles]
size_t ws_bytes_for(int B, int T, int Hv, int packed) {
  const size_t table = align_up(sizeof(int32_t) * ((size_t)B + 1), 256);
  return 256 + table + (size_t)num_slots(B, T, packed) * Hv * gdn::kWsPerSlotHead;
}

int set_cuda_error(cudaError_t e, int code) {
  t_last_cuda_error = (int)e;
  return code;
}

// Grow-only buffer for the current device.  Freeing synchronises the device.
int ensure(void*& ptr, size_t& have, size_t need) {
  if (need <= have) return GDN_OK;
  if (ptr != nullptr) {
    cudaError_t e = cudaFree(ptr);
    ptr = nullptr;
    have = 0;
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_ALLOC);
  }
  size_t want = align_up(need, (size_t)1 << 21);
  cudaError_t e = cudaMalloc(&ptr, want);
  if (e != cudaSuccess) {
    ptr = nullptr;
    (void)cudaGetLastError();
    return set_cuda_error(e, GDN_ERR_ALLOC);
  }
  have = want;
  return GDN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int launch_all(const void* q, const void* k, const void* v, const float* g, const float* beta,
               const int32_t* cu, const float* init, void* out, float* fin, int B, int T, int Hk, int Hv,
               int dk, int dv, cudaStream_t st, void* ws, int norm_qk = 0) {
  const int packed = cu != nullptr;
  int* err = static_cast<int*>(ws);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) + 256);
  void* tiles = static_cast<unsigned char*>(ws) + 256 + align_up(sizeof(int32_t) * ((size_t)B + 1), 256);
  const int nc_dense = (T + gdn::kChunk - 1) / gdn::kChunk;
  const long long nslots = num_slots(B, T, packed);
  cudaError_t e = cudaSuccess;
  if (packed) {
    e = gdn::launch_chunk_table(cu, B, T, chunk_off, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  cudaEvent_t ev[3] = {t_phase_ev[0], t_phase_ev[1], t_phase_ev[2]};
  t_phase_ev[0] = t_phase_ev[1] = t_phase_ev[2] = nullptr;
  if (ev[0] != nullptr && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (nslots > 0) {
    if (nslots > 0x7fffffffLL) return GDN_ERR_ARG;
    switch (dk) {
      case 32: e = gdn::launch_prep<32>(q, k, g, beta, cu, chunk_off, tiles, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, st); break;
      case 64: e = gdn::launch_prep<64>(q, k, g, beta, cu, chunk_off, tiles, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, st); break;
      default: e = gdn::launch_prep<128>(q, k, g, beta, cu, chunk_off, tiles, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, st); break;
    }
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  if (ev[1] != nullptr && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  switch (dk) {
    case 32: e = gdn::launch_chain_tc<32>(q, k, v, g, beta, cu, chunk_off, tiles, init, out, fin, err, B, T, Hk, Hv, dv, nc_dense, nslots, norm_qk, st); break;
    case 64: e = gdn::launch_chain_tc<64>(q, k, v, g, beta, cu, chunk_off, tiles, init, out, fin, err, B, T, Hk, Hv, dv, nc_dense, nslots, norm_qk, st); break;
    default: e = gdn::launch_chain_tc<128>(q, k, v, g, beta, cu, chunk_off, tiles, init, out, fin, err, B, T, Hk, Hv, dv, nc_dense, nslots, norm_qk, st); break;
  }
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (ev[2] != nullptr && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

}  // namespace

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

const char* gdn_strerror(int status) {
  switch (status) {
    case GDN_OK: return "ok";
    case GDN_ERR_ARG: return "invalid argument (null pointer, size, head ratio or unsupported dk/dv)";
    case GDN_ERR_ALIGN: return "pointer not 16-byte aligned";
    case GDN_ERR_ALLOC: return "device workspace allocation failed";
    case GDN_ERR_LAUNCH: return "CUDA launch or runtime call failed";
    case GDN_ERR_SCRATCH: return "problem needs more scratch than the fixed or caller-given workspace";
    default: return "unknown status";
  }
}

int gdn_last_cuda_error(void) { return t_last_cuda_error; }

void gdn_set_phase_events(void* ev_begin, void* ev_mid, void* ev_end) {
  t_phase_ev[0] = static_cast<cudaEvent_t>(ev_begin);
  t_phase_ev[1] = static_cast<cudaEvent_t>(ev_mid);
  t_phase_ev[2] = static_cast<cudaEvent_t>(ev_end);
}

size_t gdn_workspace_bytes(int B, int T, int Hk, int Hv, int dk, int dv, int packed) {
  if (check_sizes(B, T, Hk, Hv, dk, dv) != GDN_OK) return 0;
  return ws_bytes_for(B, T, Hv, packed);
}

int gdn_prefill(const void* q, const void* k, const void* v, const float* g, const float* beta,
                const int32_t* cu_seqlens, const float* init_state, void* out, float* final_state, int B,
                int T, int Hk, int Hv, int dk, int dv, void* stream) {
  t_last_cuda_error = 0;
  int rc = check_sizes(B, T, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  const long long ntok = cu_seqlens != nullptr ? (long long)T : (long long)B * T;
  if (ntok > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
  if (ntok > 0x7fffffffLL) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, init_state, out, final_state};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return GDN_ERR_ALIGN;
  if (ntok == 0 && final_state == nullptr) return GDN_OK;

  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_ARG;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hv, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    ws = d.ws;
  }
  return launch_all(q, k, v, g, beta, cu_seqlens, init_state, out, final_state, B, T, Hk, Hv, dk, dv,
                    static_cast<cudaStream_t>(stream), ws);
}

int gdn_prefill_ws(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const float* init_state, void* out, float* final_state, int B,
                   int T, int Hk, int Hv, int dk, int dv, void* workspace, size_t workspace_bytes,
                   void* stream) {
  t_last_cuda_error = 0;
  int rc = check_sizes(B, T, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  const long long ntok = cu_seqlens != nullptr ? (long long)T : (long long)B * T;
  if (ntok > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
  if (ntok > 0x7fffffffLL) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, init_state, out, final_state};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return GDN_ERR_ALIGN;
  if (ntok == 0 && final_state == nullptr) return GDN_OK;
  if (workspace == nullptr) return GDN_ERR_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return GDN_ERR_ALIGN;
  if (workspace_bytes < ws_bytes_for(B, T, Hv, cu_seqlens != nullptr)) return GDN_ERR_SCRATCH;
  return launch_all(q, k, v, g, beta, cu_seqlens, init_state, out, final_state, B, T, Hk, Hv, dk, dv,
                    static_cast<cudaStream_t>(stream), workspace);
}

int gdn_decode(const void* q, const void* k, const void* v, const float* g, const float* beta, float* state,
               void* out, int B, int Hk, int Hv, int dk, int dv, void* stream) {
  t_last_cuda_error = 0;
  int rc = check_sizes(B, 1, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  if ((long long)B * Hv > 0x7fffffffLL) return GDN_ERR_ARG;
  if (!q || !k || !v || !g || !beta || !state || !out) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, state, out};
  for (const void* p : ptrs)
    if (!aligned16(p)) return GDN_ERR_ALIGN;
  cudaError_t e;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  switch (dk) {
    case 32: e = gdn::launch_decode<32>(q, k, v, g, beta, state, out, B, Hk, Hv, dv, st); break;
    case 64: e = gdn::launch_decode<64>(q, k, v, g, beta, state, out, B, Hk, Hv, dv, st); break;
    default: e = gdn::launch_decode<128>(q, k, v, g, beta, state, out, B, Hk, Hv, dv, st); break;
  }
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

int gdn_prefill_ex(const void* q, const void* k, const void* v, const float* g, const float* beta,
                   const int32_t* cu_seqlens, const float* init_state, void* out, float* final_state, int B,
                   int T, int Hk, int Hv, int dk, int dv, unsigned flags, void* stream) {
  t_last_cuda_error = 0;
  if ((flags & ~(unsigned)GDN_FLAG_L2NORM_QK) != 0) return GDN_ERR_ARG;
  int rc = check_sizes(B, T, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  const long long ntok = cu_seqlens != nullptr ? (long long)T : (long long)B * T;
  if (ntok > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
  if (ntok > 0x7fffffffLL) return GDN_ERR_ARG;
  const void* ptrs[] = {q, k, v, g, beta, cu_seqlens, init_state, out, final_state};
  for (const void* p : ptrs)
    if (p != nullptr && !aligned16(p)) return GDN_ERR_ALIGN;
  if (ntok == 0 && final_state == nullptr) return GDN_OK;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_ARG;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hv, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    ws = d.ws;
  }
  return launch_all(q, k, v, g, beta, cu_seqlens, init_state, out, final_state, B, T, Hk, Hv, dk, dv,
                    static_cast<cudaStream_t>(stream), ws, (flags & GDN_FLAG_L2NORM_QK) ? 1 : 0);
}

int gdn_prefill_host(const void* q, const void* k, const void* v, const float* g, const float* beta,
                     const int32_t* cu_seqlens, const float* init_state, void* out, float* final_state, int B,
                     int T, int Hk, int Hv, int dk, int dv, void* stream) {
  t_last_cuda_error = 0;
  int rc = check_sizes(B, T, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if (B == 0) return GDN_OK;
  const size_t ntok = cu_seqlens != nullptr ? (size_t)T : (size_t)B * T;
  if (ntok > 0 && (!q || !k || !v || !g || !beta || !out)) return GDN_ERR_ARG;
  if (ntok > 0x7fffffffULL) return GDN_ERR_ARG;
  const size_t nq = ntok * Hk * dk * 2, nv = ntok * Hv * dv * 2, ng = ntok * Hv * 4;
  const size_t ncu = cu_seqlens ? sizeof(int32_t) * ((size_t)B + 1) : 0;
  const size_t ns = (size_t)B * Hv * dv * dk * 4;
  size_t off[9], total = 0;
  const size_t sz[9] = {nq, nq, nv, ng, ng, ncu, init_state ? ns : 0, nv, final_state ? ns : 0};
  for (int i = 0; i < 9; ++i) {
    off[i] = total;
    total += align_up(sz[i], 256);
  }
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_ARG;
  unsigned char* base = nullptr;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    rc = ensure(d.stage, d.stage_bytes, total);
    if (rc != GDN_OK) return rc;
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hv, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    base = static_cast<unsigned char*>(d.stage);
    ws = d.ws;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const void* src[7] = {q, k, v, g, beta, cu_seqlens, init_state};
  for (int i = 0; i < 7; ++i) {
    if (sz[i] == 0 || src[i] == nullptr) continue;
    e = cudaMemcpyAsync(base + off[i], src[i], sz[i], cudaMemcpyHostToDevice, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  auto P = [&](int i) -> void* { return sz[i] ? base + off[i] : nullptr; };
  rc = launch_all(P(0), P(1), P(2), static_cast<const float*>(P(3)), static_cast<const float*>(P(4)),
                  cu_seqlens ? static_cast<const int32_t*>(P(5)) : nullptr,
                  init_state ? static_cast<const float*>(P(6)) : nullptr, P(7),
                  final_state ? static_cast<float*>(P(8)) : nullptr, B, T, Hk, Hv, dk, dv, st, ws);
  if (rc != GDN_OK) return rc;
  if (nv) {
    e = cudaMemcpyAsync(out, P(7), nv, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  if (final_state) {
    e = cudaMemcpyAsync(final_state, P(8), ns, cudaMemcpyDeviceToHost, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

int gdn_device_status(int* status) {
  t_last_cuda_error = 0;
  if (status == nullptr) return GDN_ERR_ARG;
  *status = 0;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (dev < 0 || dev >= kMaxDevices) return GDN_ERR_ARG;
  void* ws = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    ws = g_dev[dev].ws;
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (ws == nullptr) return GDN_OK;
  e = cudaMemcpy(status, ws, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  e = cudaMemset(ws, 0, sizeof(int));
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

int gdn_selftest_wait_timeout(int max_polls, int* status) {
  t_last_cuda_error = 0;
  if (status == nullptr || max_polls < 1) return GDN_ERR_ARG;
  int* d = nullptr;
  cudaError_t e = cudaMalloc(&d, sizeof(int));
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_ALLOC);
  e = cudaMemset(d, 0, sizeof(int));
  if (e == cudaSuccess) e = gdn::launch_wait_timeout_probe(max_polls, d, nullptr);
  if (e == cudaSuccess) e = cudaDeviceSynchronize();
  if (e == cudaSuccess) e = cudaMemcpy(status, d, sizeof(int), cudaMemcpyDeviceToHost);
  cudaFree(d);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

void gdn_release_workspace(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return;
  std::lock_guard<std::mutex> lock(g_mu);
  DevBuffers& d = g_dev[dev];
  cudaDeviceSynchronize();
  if (d.ws) cudaFree(d.ws);
  if (d.stage) cudaFree(d.stage);
  d = DevBuffers();
}

}  // extern "C"
