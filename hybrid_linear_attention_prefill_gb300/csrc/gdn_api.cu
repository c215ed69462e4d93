// C ABI of the chunked Gated DeltaNet prefill library: argument checks, the
// per-device workspace, and the launch sequence
//   [packed only] chunk table  ->  chunk preparation  ->  chunk-sequential state carry.
// The interface style -- a versioned C ABI, scratch owned by the library and
// only ever grown, oversize or malformed requests refused before any work --
// follows the pages' native CUDA library ("Cua-S1 4B 0.2 native text worker",
// CUDA Graph paragraph; "Open-Jev-27B-v1.1 native text worker", "Build and
// serve" and "Prepare the checkpoint").
#include <algorithm>
#include <atomic>
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
template <int DK>
cudaError_t launch_chain_tc(const void*, const void*, const void*, const float*, const float*, const int32_t*,
                            const int32_t*, const int32_t*, const void*, const float*, const float*, void*, float*,
                            int*, int, int, int, int, int, int, long long, int, int, int, int, int, int,
                            cudaStream_t);
template <int DK>
cudaError_t launch_chain_f16(const void*, const float*, const float*, const int32_t*, const int32_t*,
                             const int32_t*, const void*, const void*, const float*, void*, float*, int*, int, int,
                             int, int, int, int, long long, int, int, int, int, int, int, cudaStream_t);
cudaError_t launch_wait_timeout_probe(int max_polls, int* status, cudaStream_t st);
cudaError_t launch_seg_setup(const float*, float*, float*, int32_t*, int32_t*, int, int, int, int, int, int, int,
                             cudaStream_t);
cudaError_t launch_seg_combine(const float*, const float*, const float*, float*, int, int, int, int, int,
                               cudaStream_t);
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
  void* scan = nullptr;   // two-level scan buffers (its first bytes: an all-zero value tensor)
  size_t scan_bytes = 0;
  size_t scan_zeroed = 0;
  cudaStream_t aux = nullptr;  // second stream for pass A's transition run
  cudaEvent_t fork = nullptr, join = nullptr;
  int sms = 0;
  // gdn_prefill_host's copy / compute pipeline over head groups or token windows
  bool pipe_ready = false;
  cudaStream_t h2d = nullptr, d2h = nullptr, comp[3] = {nullptr, nullptr, nullptr};
  cudaEvent_t ev_start = nullptr, ev_end = nullptr, ev_in[8] = {}, ev_prep[8] = {}, ev_done[8] = {};
};

constexpr int kMaxHostGroups = 4;   // head groups (packed batches)
constexpr int kMaxHostWindows = 8;      // token windows (dense batches)
constexpr int kHostWindowChunks = 16;   // chunks per window, about (measured best over 2..16 windows)

std::mutex g_mu;
DevBuffers g_dev[kMaxDevices];
thread_local int t_last_cuda_error = 0;
thread_local cudaEvent_t t_phase_ev[3] = {nullptr, nullptr, nullptr};
std::atomic<int> g_fail_allocs{0};  // gdn_debug_fail_allocations

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

// Workspace: [256 B status words][chunk table and dispatch order (chunk_table_bytes)]
//            [Tm/PT tiles per (slot, value head)][inverse q/k norms per (slot, key head)]
//            [fp16 [K; Q] images per (slot, key head)]
size_t ws_bytes_for(int B, int T, int Hk, int Hv, int dk, int packed) {
  const size_t table = gdn::chunk_table_bytes(B);
  const size_t ns = (size_t)num_slots(B, T, packed);
  return 256 + table + ns * Hv * gdn::kWsPerSlotHead + ns * Hk * gdn::kWsNormPerSlotKHead +
         ns * Hk * gdn::kws_kq_bytes(dk);
}

using gdn::set_cuda_error;

// Grow-only buffer for the current device.  Freeing synchronises the device.  An
// injected failure (gdn_debug_fail_allocations) fails before anything is freed, so
// the old buffer stays usable.
int ensure(void*& ptr, size_t& have, size_t need) {
  if (need <= have) return GDN_OK;
  if (gdn::take_injected_alloc_failure()) return set_cuda_error(cudaErrorMemoryAllocation, GDN_ERR_ALLOC);
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

// ---- two-level chunk scan (dense batches with few heads and many chunks) -----------
// Number of segments P (1 = the single-level path).  Pass A runs, at once, the
// zero-start carry of segments 0 .. B P - 2 (dv / 32 CTAs per head each) and the
// transition carry of segments 1 .. B P - 2 (dk / 32 per head), so P is the largest
// count whose pass A fits one wave on the device's SMs -- at least 3 (with 2 the two
// passes take as long as one unsegmented pass) and at most one segment per 8 chunks.
int choose_segments(int B, int T, int Hv, int dk, int dv, bool packed, unsigned flags, int sms) {
  if (packed || (flags & GDN_FLAG_ONE_LEVEL) != 0 || B <= 0 || T <= 0) return 1;
  const long long nc = (T + gdn::kChunk - 1) / gdn::kChunk;
  // Hv ((B P - 1) dv + (B P - 2) dk) / 32 <= sms
  const long long fit = ((long long)sms * 32 / std::max(Hv, 1) + dv + 2LL * dk) / ((long long)B * (dv + dk));
  const int req = (int)((flags >> 8) & 0xffu);
  if ((flags & GDN_FLAG_TWO_LEVEL) != 0) {
    long long P = req >= 2 ? req : std::max<long long>(3, fit);
    P = std::min(P, nc);
    return P >= 2 ? (int)P : 1;
  }
  // segments of at least 8 chunks, so the two passes beat one by more than the
  // set-up and combine cost
  long long P = std::min<long long>(std::min<long long>(fit, nc / 8), 32);
  return P >= 3 ? (int)P : 1;
}

struct ScanLayout {
  size_t vzero, oscr, cu, off, a_init, i_init, n_fin, phi, c_init, f_fin, total;
};

ScanLayout scan_layout(int B, int T, int Hv, int dk, int dv, int P) {
  ScanLayout L;
  const size_t ntok = (size_t)B * T, bp = (size_t)B * P;
  const size_t st = bp * Hv * dv * dk * 4, sp = bp * Hv * dk * dk * 4;
  size_t o = 0;
  auto take = [&](size_t n) { const size_t r = o; o += align_up(n, 256); return r; };
  L.vzero = take(ntok * Hv * dk * 2);  // first, so the zeroed prefix only ever grows
  L.oscr = take(ntok * Hv * dk * 2);
  L.cu = take((bp + 1) * 4);
  L.off = take((bp + 1) * 4);
  L.a_init = take(st);
  L.i_init = take(sp);
  L.n_fin = take(st);
  L.phi = take(sp);
  L.c_init = take(st);
  L.f_fin = take(st);
  L.total = o;
  return L;
}

struct ScanPlan {
  int P = 1;
  unsigned char* buf = nullptr;
  cudaStream_t aux = nullptr;
  cudaEvent_t fork = nullptr, join = nullptr;
};

// Segment count and (when P > 1) buffers, stream and events for the calling device.
int prepare_scan(int dev, int B, int T, int Hv, int dk, int dv, bool packed, unsigned flags, cudaStream_t st,
                 ScanPlan& plan) {
  DevBuffers& d = g_dev[dev];
  if (d.sms == 0) {
    cudaError_t e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  plan.P = choose_segments(B, T, Hv, dk, dv, packed, flags, d.sms);
  if (plan.P <= 1) return GDN_OK;
  const ScanLayout L = scan_layout(B, T, Hv, dk, dv, plan.P);
  void* before = d.scan;
  int rc = ensure(d.scan, d.scan_bytes, L.total);
  if (rc != GDN_OK) return rc;
  if (d.scan != before) d.scan_zeroed = 0;  // a new allocation
  if (L.oscr > d.scan_zeroed) {  // the zero value tensor of the transition run
    cudaError_t e = cudaMemsetAsync(d.scan, 0, L.oscr, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  // this call writes its scratch outputs right after the zero tensor, so only that
  // tensor is known to be zero afterwards
  d.scan_zeroed = L.oscr;
  if (d.aux == nullptr) {
    cudaError_t e = cudaStreamCreateWithFlags(&d.aux, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.fork, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.join, cudaEventDisableTiming);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  plan.buf = static_cast<unsigned char*>(d.scan);
  plan.aux = d.aux;
  plan.fork = d.fork;
  plan.join = d.join;
  return GDN_OK;
}

// The state carry of value heads [h_base, h_base + h_count): fp16 operands by default, bf16
// hi / lo pairs when `wide` (then with q and k read from the inputs).  check_small: the fp16
// kernel reports a final state below its accurate range (off for the two-level scan's runs).
template <int DK>
cudaError_t carry(int wide, const void* q, const void* k, const void* v, const float* g, const float* beta,
                  const int32_t* cu, const int32_t* chunk_off, const int32_t* order, const void* tiles,
                  const float* ws_rn, const void* ws_kq, const float* init, void* out, float* fin, int* err, int B,
                  int T, int Hk, int Hv, int DV, int nc_dense, long long nslots, int norm_qk, int h_base,
                  int h_count, int c_begin, int c_end, int slice, int check_small, cudaStream_t st) {
  if (wide)
    return gdn::launch_chain_tc<DK>(q, k, v, g, beta, cu, chunk_off, order, tiles, ws_rn, init, out, fin, err, B, T,
                                    Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end, slice, st);
  return gdn::launch_chain_f16<DK>(v, g, beta, cu, chunk_off, order, tiles, ws_kq, init, out, fin, err, B, T, Hk,
                                   Hv, DV, nc_dense, nslots, h_base, h_count, c_begin, c_end, slice, check_small, st);
}

cudaError_t carry_dk(int dk, int wide, const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const int32_t* cu, const int32_t* chunk_off, const int32_t* order,
                     const void* tiles, const float* ws_rn, const void* ws_kq, const float* init, void* out,
                     float* fin, int* err, int B, int T, int Hk, int Hv, int DV, int nc_dense, long long nslots,
                     int norm_qk, int h_base, int h_count, int c_begin, int c_end, int slice, int check_small,
                     cudaStream_t st) {
  switch (dk) {
    case 32: return carry<32>(wide, q, k, v, g, beta, cu, chunk_off, order, tiles, ws_rn, ws_kq, init, out, fin, err, B, T, Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end, slice, check_small, st);
    case 64: return carry<64>(wide, q, k, v, g, beta, cu, chunk_off, order, tiles, ws_rn, ws_kq, init, out, fin, err, B, T, Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end, slice, check_small, st);
    default: return carry<128>(wide, q, k, v, g, beta, cu, chunk_off, order, tiles, ws_rn, ws_kq, init, out, fin, err, B, T, Hk, Hv, DV, nc_dense, nslots, norm_qk, h_base, h_count, c_begin, c_end, slice, check_small, st);
  }
}

// A run of the two-level scan.  Its runs are packed views of segments: dispatched in their own
// order, with 32 state rows per CTA (its choice of the segment count counts 32-row CTAs, so that
// pass A's two runs fit one wave side by side).
cudaError_t chain_dk(int dk, int wide, const void* q, const void* k, const void* v, const float* g,
                     const float* beta, const int32_t* cu, const int32_t* chunk_off, const void* tiles,
                     const float* ws_rn, const void* ws_kq, const float* init, void* out, float* fin, int* err,
                     int B, int T, int Hk, int Hv, int DV, int nc_dense, long long nslots, int norm_qk,
                     cudaStream_t st) {
  return carry_dk(dk, wide, q, k, v, g, beta, cu, chunk_off, nullptr, tiles, ws_rn, ws_kq, init, out, fin, err, B, T,
                  Hk, Hv, DV, nc_dense, nslots, norm_qk, 0, Hv, 0, INT_MAX, 32, 0, st);
}

// The prefill for value heads [h0, h1) (all heads when h1 < 0; h0 and h1 multiples of
// Hv / Hk) on `st`.  `table` = false skips the packed chunk table (already built).
int launch_all(const void* q, const void* k, const void* v, const float* g, const float* beta,
               const int32_t* cu, const float* init, void* out, float* fin, int B, int T, int Hk, int Hv,
               int dk, int dv, cudaStream_t st, void* ws, int norm_qk = 0, const ScanPlan* plan = nullptr,
               int h0 = 0, int h1 = -1, bool table = true, int c0 = 0, int c1 = -1, int phases = 3,
               int slice = 0, int wide = 0) {
  // [h0, h1): value heads; [c0, c1): the window of each dense sequence's chunks (-1: all).
  // A window's launches carry the state from `init` to `fin` over its chunks only.
  // phases: bit 0 the preparation kernel (and the packed chunk table), bit 1 the state carry.
  // slice: state rows per state-carry CTA (16, 32, 64; 0 = the library's choice).
  // wide: the bf16 hi / lo state carry (fp32 range) instead of the fp16 one.
  if (h1 < 0) h1 = Hv;
  const int G = Hv / Hk;
  const int hk0 = h0 / G, nhk = (h1 - h0) / G;
  const int packed = cu != nullptr;
  int* err = static_cast<int*>(ws);
  int32_t* chunk_off = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) + 256);
  int32_t* order = packed ? chunk_off + B + 1 : nullptr;  // packed: state carries longest first
  void* tiles = static_cast<unsigned char*>(ws) + 256 + gdn::chunk_table_bytes(B);
  const int nc_dense = (T + gdn::kChunk - 1) / gdn::kChunk;
  const long long nslots = num_slots(B, T, packed);
  if (c1 < 0) c1 = nc_dense;
  const bool whole = c0 == 0 && c1 == nc_dense;
  if (!packed && (c0 < 0 || c1 > nc_dense || c0 >= c1) && nc_dense > 0) return GDN_ERR_ARG;
  const int cc0 = packed ? 0 : c0, cc1 = packed ? INT_MAX : c1;  // the chain's window
  // a whole problem's preparation kernel has the device to itself; a piece of the host
  // entry's pipeline runs beside other pieces' kernels
  const int alone = whole && h0 == 0 && h1 == Hv && phases == 3;
  float* ws_rn = reinterpret_cast<float*>(static_cast<unsigned char*>(tiles) + (size_t)nslots * Hv * gdn::kWsPerSlotHead);
  void* ws_kq = reinterpret_cast<unsigned char*>(ws_rn) + (size_t)nslots * Hk * gdn::kWsNormPerSlotKHead;
  cudaError_t e = cudaSuccess;
  if (packed && table && (phases & 1)) {
    e = gdn::launch_chunk_table(cu, B, T, chunk_off, order, err, st);
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  cudaEvent_t ev[3];
  gdn::take_phase_events(ev);
  if (ev[0] != nullptr && (e = cudaEventRecord(ev[0], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (nslots > 0x7fffffffLL) return GDN_ERR_ARG;
  if (nslots > 0 && (phases & 1)) {
    switch (dk) {
      case 32: e = gdn::launch_prep<32>(q, k, g, beta, cu, chunk_off, tiles, ws_rn, ws_kq, !wide, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, hk0, nhk, c0, c1 - c0, alone, st); break;
      case 64: e = gdn::launch_prep<64>(q, k, g, beta, cu, chunk_off, tiles, ws_rn, ws_kq, !wide, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, hk0, nhk, c0, c1 - c0, alone, st); break;
      default: e = gdn::launch_prep<128>(q, k, g, beta, cu, chunk_off, tiles, ws_rn, ws_kq, !wide, err, B, T, Hk, Hv, (int)nslots, nc_dense, norm_qk, hk0, nhk, c0, c1 - c0, alone, st); break;
    }
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  }
  if (ev[1] != nullptr && (e = cudaEventRecord(ev[1], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (!(phases & 2)) return GDN_OK;
  if (plan != nullptr && plan->P > 1 && !packed && nslots > 0 && h0 == 0 && h1 == Hv && whole) {
    // ---- two-level scan over P segments per sequence (see gdn_scan.cu) ----------------
    const int P = plan->P, BP = B * P;
    const int cps = (nc_dense + P - 1) / P;  // chunks per segment
    const ScanLayout L = scan_layout(B, T, Hv, dk, dv, P);
    unsigned char* sb = plan->buf;
    void* vzero = sb + L.vzero;
    void* oscr = sb + L.oscr;
    int32_t* cu_seg = reinterpret_cast<int32_t*>(sb + L.cu);
    int32_t* off_seg = reinterpret_cast<int32_t*>(sb + L.off);
    float* a_init = reinterpret_cast<float*>(sb + L.a_init);
    float* i_init = reinterpret_cast<float*>(sb + L.i_init);
    float* n_fin = reinterpret_cast<float*>(sb + L.n_fin);
    float* phi = reinterpret_cast<float*>(sb + L.phi);
    float* c_init = reinterpret_cast<float*>(sb + L.c_init);
    float* f_fin = reinterpret_cast<float*>(sb + L.f_fin);
    const int ttot = B * T;
    if ((e = gdn::launch_seg_setup(init, a_init, i_init, cu_seg, off_seg, B, T, P, cps, Hv, dv, dk, st)) !=
            cudaSuccess ||
        (e = cudaEventRecord(plan->fork, st)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(plan->aux, plan->fork, 0)) != cudaSuccess)
      return set_cuda_error(e, GDN_ERR_LAUNCH);
    // Each run below covers a contiguous range [first, first + n) of the segment list,
    // passed as a packed batch of n sequences by offsetting cu_seg, off_seg and the
    // per-sequence init / final-state pointers.  Segments a run does not need (the
    // last of each sequence in the zero-start run, the first in pass C, ...) are left
    // out wherever they sit at the ends of the list.
    const size_t ps = (size_t)Hv * dv * dk, pi = (size_t)Hv * dk * dk;
    // pass A: zero-start runs of segments 0 .. BP-2 (segment 0 of each sequence from the
    // true initial state: its outputs are final) beside the transition runs of 1 .. BP-2
    // (v = 0 from the identity, dk rows) on the second stream
    if (BP - 2 >= 1 &&
        (e = chain_dk(dk, wide, q, k, vzero, g, beta, cu_seg + 1, off_seg + 1, tiles, ws_rn, ws_kq, i_init + pi, oscr,
                      phi + pi, err, BP - 2, ttot, Hk, Hv, dk, nc_dense, nslots, norm_qk, plan->aux)) != cudaSuccess)
      return set_cuda_error(e, GDN_ERR_LAUNCH);
    if ((e = chain_dk(dk, wide, q, k, v, g, beta, cu_seg, off_seg, tiles, ws_rn, ws_kq, a_init, out, n_fin, err, BP - 1,
                      ttot, Hk, Hv, dv, nc_dense, nslots, norm_qk, st)) != cudaSuccess ||
        (e = cudaEventRecord(plan->join, plan->aux)) != cudaSuccess ||
        (e = cudaStreamWaitEvent(st, plan->join, 0)) != cudaSuccess)
      return set_cuda_error(e, GDN_ERR_LAUNCH);
    // segment start states, then pass C over segments 1 .. BP-1 (the outputs; the last
    // segment's final state)
    if ((e = gdn::launch_seg_combine(init, n_fin, phi, c_init, B, P, Hv, dv, dk, st)) != cudaSuccess ||
        (e = chain_dk(dk, wide, q, k, v, g, beta, cu_seg + 1, off_seg + 1, tiles, ws_rn, ws_kq, c_init + ps, out,
                      f_fin + ps, err, BP - 1, ttot, Hk, Hv, dv, nc_dense, nslots, norm_qk, st)) != cudaSuccess)
      return set_cuda_error(e, GDN_ERR_LAUNCH);
    if (fin != nullptr) {
      const size_t per = (size_t)Hv * dv * dk;
      for (int b = 0; b < B; ++b) {
        e = cudaMemcpyAsync(fin + (size_t)b * per, f_fin + ((size_t)b * P + P - 1) * per, per * sizeof(float),
                            cudaMemcpyDeviceToDevice, st);
        if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
      }
    }
    if (ev[2] != nullptr && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
    return GDN_OK;
  }
  e = carry_dk(dk, wide, q, k, v, g, beta, cu, chunk_off, order, tiles, ws_rn, ws_kq, init, out, fin, err, B, T, Hk,
               Hv, dv, nc_dense, nslots, norm_qk, h0, h1 - h0, cc0, cc1, slice, 1, st);
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  if (ev[2] != nullptr && (e = cudaEventRecord(ev[2], st)) != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  return GDN_OK;
}

}  // namespace

namespace gdn {

int set_cuda_error(cudaError_t e, int code) {
  t_last_cuda_error = (int)e;
  return code;
}

void clear_cuda_error() { t_last_cuda_error = 0; }

void take_phase_events(cudaEvent_t (&ev)[3]) {
  for (int i = 0; i < 3; ++i) {
    ev[i] = t_phase_ev[i];
    t_phase_ev[i] = nullptr;
  }
}

bool take_injected_alloc_failure() {
  int n = g_fail_allocs.load();
  while (n > 0 && !g_fail_allocs.compare_exchange_weak(n, n - 1)) {
  }
  return n > 0;
}

}  // namespace gdn

extern "C" {

int gdn_abi_version(void) { return GDN_ABI_VERSION; }

int gdn_debug_fail_allocations(int count) { return g_fail_allocs.exchange(count < 0 ? 0 : count); }

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

int gdn_scan_segments(int B, int T, int Hk, int Hv, int dk, int dv, int packed, unsigned flags) {
  const unsigned known =
      GDN_FLAG_L2NORM_QK | GDN_FLAG_TWO_LEVEL | GDN_FLAG_ONE_LEVEL | 0xff00u | GDN_FLAG_SLICE16 | GDN_FLAG_SLICE32 |
      GDN_FLAG_SLICE64 | GDN_FLAG_WIDE_RANGE;
  if (check_sizes(B, T, Hk, Hv, dk, dv) != GDN_OK || (flags & ~known) != 0) return 0;
  if ((flags & GDN_FLAG_TWO_LEVEL) && (flags & GDN_FLAG_ONE_LEVEL)) return 0;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
    (void)cudaGetLastError();
    return 0;
  }
  return choose_segments(B, T, Hv, dk, dv, packed != 0, flags, sms);
}

size_t gdn_workspace_bytes(int B, int T, int Hk, int Hv, int dk, int dv, int packed) {
  if (check_sizes(B, T, Hk, Hv, dk, dv) != GDN_OK) return 0;
  return ws_bytes_for(B, T, Hk, Hv, dk, packed);
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
  ScanPlan plan;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hk, Hv, dk, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    ws = d.ws;
    rc = prepare_scan(dev, B, T, Hv, dk, dv, cu_seqlens != nullptr, 0u, static_cast<cudaStream_t>(stream), plan);
    if (rc != GDN_OK) return rc;
  }
  return launch_all(q, k, v, g, beta, cu_seqlens, init_state, out, final_state, B, T, Hk, Hv, dk, dv,
                    static_cast<cudaStream_t>(stream), ws, 0, &plan);
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
  if (workspace_bytes < ws_bytes_for(B, T, Hk, Hv, dk, cu_seqlens != nullptr)) return GDN_ERR_SCRATCH;
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
  const unsigned known =
      GDN_FLAG_L2NORM_QK | GDN_FLAG_TWO_LEVEL | GDN_FLAG_ONE_LEVEL | 0xff00u | GDN_FLAG_SLICE16 | GDN_FLAG_SLICE32 |
      GDN_FLAG_SLICE64 | GDN_FLAG_WIDE_RANGE;
  if ((flags & ~known) != 0) return GDN_ERR_ARG;
  if ((flags & GDN_FLAG_TWO_LEVEL) && (flags & GDN_FLAG_ONE_LEVEL)) return GDN_ERR_ARG;
  {
    const unsigned sl = flags & (GDN_FLAG_SLICE16 | GDN_FLAG_SLICE32 | GDN_FLAG_SLICE64);
    if (sl & (sl - 1)) return GDN_ERR_ARG;  // at most one slice width
  }
  int rc = check_sizes(B, T, Hk, Hv, dk, dv);
  if (rc != GDN_OK) return rc;
  if ((flags & GDN_FLAG_SLICE64) && dv % 64 != 0) return GDN_ERR_ARG;
  const int slice =
      (flags & GDN_FLAG_SLICE16) ? 16 : (flags & GDN_FLAG_SLICE32) ? 32 : (flags & GDN_FLAG_SLICE64) ? 64 : 0;
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
  ScanPlan plan;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hk, Hv, dk, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    ws = d.ws;
    rc = prepare_scan(dev, B, T, Hv, dk, dv, cu_seqlens != nullptr, flags, static_cast<cudaStream_t>(stream), plan);
    if (rc != GDN_OK) return rc;
  }
  return launch_all(q, k, v, g, beta, cu_seqlens, init_state, out, final_state, B, T, Hk, Hv, dk, dv,
                    static_cast<cudaStream_t>(stream), ws, (flags & GDN_FLAG_L2NORM_QK) ? 1 : 0, &plan, 0, -1, true,
                    0, -1, 3, slice, (flags & GDN_FLAG_WIDE_RANGE) ? 1 : 0);
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
  // the state slot also carries the state between token windows of a dense batch
  const size_t sz[9] = {nq, nq, nv, ng, ng, ncu, init_state ? ns : 0, nv,
                        (final_state != nullptr || cu_seqlens == nullptr) ? ns : 0};
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
  ScanPlan plan;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  DevBuffers* dp = nullptr;
  // Dense batches: token windows of whole chunks.  The copies of window i + 1 overlap the
  // kernels of window i and the copy-out of earlier windows; each window's state carry
  // starts from the state the previous one left, so the tail after the last copy-in is
  // one window's kernels and copy-out.  Packed batches: head groups, whose copies of group
  // i + 1 overlap the kernels of group i (each group on its own stream, so the
  // latency-bound state carries of all groups run side by side).  Whole key heads per
  // group.  One piece for small problems or with the two-level scan.
  int ngroups = 1, nwin = 1;
  const int nc_dense = (T + gdn::kChunk - 1) / gdn::kChunk;
  {
    std::lock_guard<std::mutex> lock(g_mu);
    DevBuffers& d = g_dev[dev];
    dp = &d;
    rc = ensure(d.stage, d.stage_bytes, total);
    if (rc != GDN_OK) return rc;
    rc = ensure(d.ws, d.ws_bytes, ws_bytes_for(B, T, Hk, Hv, dk, cu_seqlens != nullptr));
    if (rc != GDN_OK) return rc;
    base = static_cast<unsigned char*>(d.stage);
    ws = d.ws;
    rc = prepare_scan(dev, B, T, Hv, dk, dv, cu_seqlens != nullptr, 0u, st, plan);
    if (rc != GDN_OK) return rc;
    if (plan.P <= 1 && nq + nv >= ((size_t)8 << 20)) {
      if (cu_seqlens == nullptr)
        nwin = nc_dense < 2 ? 1 : std::min(kMaxHostWindows, std::max(2, nc_dense / kHostWindowChunks));
      else
        ngroups = std::min(kMaxHostGroups, Hk);
    }
    if ((ngroups > 1 || nwin > 1) && !d.pipe_ready) {
      e = cudaStreamCreateWithFlags(&d.h2d, cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&d.d2h, cudaStreamNonBlocking);
      for (int i = 0; i < 3 && e == cudaSuccess; ++i) e = cudaStreamCreateWithFlags(&d.comp[i], cudaStreamNonBlocking);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_start, cudaEventDisableTiming);
      if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_end, cudaEventDisableTiming);
      for (int i = 0; i < kMaxHostWindows && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&d.ev_in[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_prep[i], cudaEventDisableTiming);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&d.ev_done[i], cudaEventDisableTiming);
      }
      if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
      d.pipe_ready = true;
    }
  }
  auto P = [&](int i) -> unsigned char* { return sz[i] ? base + off[i] : nullptr; };
  const void* src[7] = {q, k, v, g, beta, cu_seqlens, init_state};
  if (ngroups <= 1 && nwin <= 1) {
    for (int i = 0; i < 7; ++i) {
      if (sz[i] == 0 || src[i] == nullptr) continue;
      e = cudaMemcpyAsync(base + off[i], src[i], sz[i], cudaMemcpyHostToDevice, st);
      if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
    }
    rc = launch_all(P(0), P(1), P(2), reinterpret_cast<const float*>(P(3)), reinterpret_cast<const float*>(P(4)),
                    cu_seqlens ? reinterpret_cast<const int32_t*>(P(5)) : nullptr,
                    init_state ? reinterpret_cast<const float*>(P(6)) : nullptr, P(7),
                    final_state ? reinterpret_cast<float*>(P(8)) : nullptr, B, T, Hk, Hv, dk, dv, st, ws, 0, &plan);
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

  DevBuffers& d = *dp;
  auto check = [&](cudaError_t x) { return x == cudaSuccess ? GDN_OK : set_cuda_error(x, GDN_ERR_LAUNCH); };
  if (nwin > 1) {
    // ---- dense: pipelined over token windows ------------------------------------------
    // tokens [ta, tb) of every sequence: B rows of (tb - ta) * row bytes, T * row bytes apart
    auto rows = [&](unsigned char* dst, const unsigned char* src_, size_t row, int ta, int tb, cudaMemcpyKind kind,
                    cudaStream_t s_) {
      return cudaMemcpy2DAsync(dst + (size_t)ta * row, (size_t)T * row, src_ + (size_t)ta * row, (size_t)T * row,
                               (size_t)(tb - ta) * row, B, kind, s_);
    };
    const size_t rq = (size_t)Hk * dk * 2, rv = (size_t)Hv * dv * 2, rg = (size_t)Hv * 4;
    const size_t rowb[5] = {rq, rq, rv, rg, rg};
    float* state = reinterpret_cast<float*>(P(8));
    cudaStream_t ps = d.comp[0];  // the preparation kernels; the state carries stay on `stream`
    if ((rc = check(cudaEventRecord(d.ev_start, st))) != GDN_OK ||
        (rc = check(cudaStreamWaitEvent(d.h2d, d.ev_start, 0))) != GDN_OK)
      return rc;
    if (init_state != nullptr &&
        (rc = check(cudaMemcpyAsync(P(6), init_state, ns, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK)
      return rc;
    // g and beta whole, first (small)
    if ((rc = check(cudaMemcpyAsync(P(3), g, ng, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK ||
        (rc = check(cudaMemcpyAsync(P(4), beta, ng, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK)
      return rc;
    for (int i = 0; i < nwin; ++i) {
      // Window weights 2, 2, ..., 2, 1: the last window is half the size of the others, so the
      // tail after the last copy-in (its kernels and copy-out) is short.  Measured e2e per step,
      // equal windows against this: T=4096 521 -> 494 us, T=16381 1733 -> 1682, T=1024 150 -> 137;
      // a further taper (4, ..., 4, 2, 1) lost at T=16381.
      const long long wsum = 2LL * nwin - 1;
      const int c0 = (int)((long long)nc_dense * (2LL * i) / wsum);
      const int c1 = i + 1 == nwin ? nc_dense : (int)((long long)nc_dense * (2LL * (i + 1)) / wsum);
      const int ta = c0 * gdn::kChunk, tb = std::min(c1 * gdn::kChunk, T);
      for (int a = 0; a < 3; ++a)
        if ((rc = check(rows(base + off[a], static_cast<const unsigned char*>(src[a]), rowb[a], ta, tb,
                             cudaMemcpyHostToDevice, d.h2d))) != GDN_OK)
          return rc;
      if ((rc = check(cudaEventRecord(d.ev_in[i], d.h2d))) != GDN_OK ||
          (rc = check(cudaStreamWaitEvent(ps, d.ev_in[i], 0))) != GDN_OK)
        return rc;
      rc = launch_all(P(0), P(1), P(2), reinterpret_cast<const float*>(P(3)), reinterpret_cast<const float*>(P(4)),
                      nullptr, nullptr, P(7), state, B, T, Hk, Hv, dk, dv, ps, ws, 0, nullptr, 0, -1, false, c0, c1,
                      1);
      if (rc != GDN_OK) return rc;
      if ((rc = check(cudaEventRecord(d.ev_prep[i], ps))) != GDN_OK ||
          (rc = check(cudaStreamWaitEvent(st, d.ev_prep[i], 0))) != GDN_OK)
        return rc;
      const float* win_init = i == 0 ? (init_state ? reinterpret_cast<const float*>(P(6)) : nullptr) : state;
      rc = launch_all(P(0), P(1), P(2), reinterpret_cast<const float*>(P(3)), reinterpret_cast<const float*>(P(4)),
                      nullptr, win_init, P(7), state, B, T, Hk, Hv, dk, dv, st, ws, 0, nullptr, 0, -1, false, c0, c1,
                      2);
      if (rc != GDN_OK) return rc;
      if ((rc = check(cudaEventRecord(d.ev_done[i], st))) != GDN_OK ||
          (rc = check(cudaStreamWaitEvent(d.d2h, d.ev_done[i], 0))) != GDN_OK ||
          (rc = check(rows(static_cast<unsigned char*>(out), P(7), rv, ta, tb, cudaMemcpyDeviceToHost, d.d2h))) !=
              GDN_OK)
        return rc;
    }
    if (final_state != nullptr &&
        (rc = check(cudaMemcpyAsync(final_state, state, ns, cudaMemcpyDeviceToHost, d.d2h))) != GDN_OK)
      return rc;
    if ((rc = check(cudaEventRecord(d.ev_end, d.d2h))) != GDN_OK ||
        (rc = check(cudaStreamWaitEvent(st, d.ev_end, 0))) != GDN_OK ||
        (rc = check(cudaStreamSynchronize(st))) != GDN_OK)
      return rc;
    return GDN_OK;
  }

  // ---- packed: pipelined over head groups ---------------------------------------------
  const int G = Hv / Hk;
  auto h2d_cols = [&](int i, size_t col0, size_t width, size_t pitch, size_t rows) {  // column band of a row-major array
    return cudaMemcpy2DAsync(base + off[i] + col0, pitch, static_cast<const unsigned char*>(src[i]) + col0, pitch,
                             width, rows, cudaMemcpyHostToDevice, d.h2d);
  };
  // the copies start after everything already queued on `stream` (earlier calls use the same staging)
  if ((rc = check(cudaEventRecord(d.ev_start, st))) != GDN_OK ||
      (rc = check(cudaStreamWaitEvent(d.h2d, d.ev_start, 0))) != GDN_OK)
    return rc;
  // small, whole: cu_seqlens (and the packed chunk table), g, beta
  if (cu_seqlens != nullptr) {
    if ((rc = check(cudaMemcpyAsync(P(5), cu_seqlens, ncu, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK) return rc;
    int32_t* chunk_off = reinterpret_cast<int32_t*>(static_cast<unsigned char*>(ws) + 256);
    if ((rc = check(gdn::launch_chunk_table(reinterpret_cast<const int32_t*>(P(5)), B, T, chunk_off,
                                            chunk_off + B + 1, static_cast<int*>(ws), d.h2d))) != GDN_OK)
      return rc;
  }
  if ((rc = check(cudaMemcpyAsync(P(3), g, ng, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK ||
      (rc = check(cudaMemcpyAsync(P(4), beta, ng, cudaMemcpyHostToDevice, d.h2d))) != GDN_OK)
    return rc;
  int hk_lo[kMaxHostGroups + 1];
  for (int i = 0; i <= ngroups; ++i) hk_lo[i] = (int)((long long)Hk * i / ngroups);
  for (int i = 0; i < ngroups; ++i) {
    const size_t k0 = (size_t)hk_lo[i], k1 = (size_t)hk_lo[i + 1];
    const size_t h0 = k0 * G, h1 = k1 * G;
    // inputs of group i: the key heads' q / k columns, the value heads' v columns, the init slices
    if ((rc = check(h2d_cols(0, k0 * dk * 2, (k1 - k0) * dk * 2, (size_t)Hk * dk * 2, ntok))) != GDN_OK ||
        (rc = check(h2d_cols(1, k0 * dk * 2, (k1 - k0) * dk * 2, (size_t)Hk * dk * 2, ntok))) != GDN_OK ||
        (rc = check(h2d_cols(2, h0 * dv * 2, (h1 - h0) * dv * 2, (size_t)Hv * dv * 2, ntok))) != GDN_OK)
      return rc;
    if (init_state != nullptr &&
        (rc = check(h2d_cols(6, h0 * dv * dk * 4, (h1 - h0) * dv * dk * 4, (size_t)Hv * dv * dk * 4, B))) != GDN_OK)
      return rc;
    if ((rc = check(cudaEventRecord(d.ev_in[i], d.h2d))) != GDN_OK) return rc;
    // kernels of group i on their own stream
    cudaStream_t cs = i == 0 ? st : d.comp[i - 1];
    if ((rc = check(cudaStreamWaitEvent(cs, d.ev_in[i], 0))) != GDN_OK) return rc;
    rc = launch_all(P(0), P(1), P(2), reinterpret_cast<const float*>(P(3)), reinterpret_cast<const float*>(P(4)),
                    cu_seqlens ? reinterpret_cast<const int32_t*>(P(5)) : nullptr,
                    init_state ? reinterpret_cast<const float*>(P(6)) : nullptr, P(7),
                    final_state ? reinterpret_cast<float*>(P(8)) : nullptr, B, T, Hk, Hv, dk, dv, cs, ws, 0, nullptr,
                    (int)h0, (int)h1, false);
    if (rc != GDN_OK) return rc;
    if ((rc = check(cudaEventRecord(d.ev_done[i], cs))) != GDN_OK) return rc;
    // outputs of group i back to the host
    if ((rc = check(cudaStreamWaitEvent(d.d2h, d.ev_done[i], 0))) != GDN_OK ||
        (rc = check(cudaMemcpy2DAsync(static_cast<unsigned char*>(out) + h0 * dv * 2, (size_t)Hv * dv * 2,
                                      P(7) + h0 * dv * 2, (size_t)Hv * dv * 2, (h1 - h0) * dv * 2, ntok,
                                      cudaMemcpyDeviceToHost, d.d2h))) != GDN_OK)
      return rc;
    if (final_state != nullptr &&
        (rc = check(cudaMemcpy2DAsync(reinterpret_cast<unsigned char*>(final_state) + h0 * dv * dk * 4,
                                      (size_t)Hv * dv * dk * 4, P(8) + h0 * dv * dk * 4, (size_t)Hv * dv * dk * 4,
                                      (h1 - h0) * dv * dk * 4, B, cudaMemcpyDeviceToHost, d.d2h))) != GDN_OK)
      return rc;
  }
  if ((rc = check(cudaEventRecord(d.ev_end, d.d2h))) != GDN_OK ||
      (rc = check(cudaStreamWaitEvent(st, d.ev_end, 0))) != GDN_OK ||
      (rc = check(cudaStreamSynchronize(st))) != GDN_OK)
    return rc;
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
  void* words[2] = {nullptr, gdn::static_scratch_address(dev)};  // the workspace's, the static array's
  {
    std::lock_guard<std::mutex> lock(g_mu);
    words[0] = g_dev[dev].ws;
  }
  e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
  for (void* w : words) {
    if (w == nullptr) continue;
    int bits = 0;
    e = cudaMemcpy(&bits, w, sizeof(int), cudaMemcpyDeviceToHost);
    if (e == cudaSuccess) e = cudaMemset(w, 0, sizeof(int));
    if (e != cudaSuccess) return set_cuda_error(e, GDN_ERR_LAUNCH);
    *status |= bits;
  }
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
  if (d.scan) cudaFree(d.scan);
  if (d.fork) cudaEventDestroy(d.fork);
  if (d.join) cudaEventDestroy(d.join);
  if (d.aux) cudaStreamDestroy(d.aux);
  if (d.pipe_ready) {
    cudaStreamDestroy(d.h2d);
    cudaStreamDestroy(d.d2h);
    for (cudaStream_t c : d.comp) cudaStreamDestroy(c);
    cudaEventDestroy(d.ev_start);
    cudaEventDestroy(d.ev_end);
    for (int i = 0; i < kMaxHostWindows; ++i) {
      cudaEventDestroy(d.ev_in[i]);
      cudaEventDestroy(d.ev_prep[i]);
      cudaEventDestroy(d.ev_done[i]);
    }
  }
  d = DevBuffers();
}

}  // extern "C"
