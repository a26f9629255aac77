// host_pipe.cu -- sa_attn_fwd_host: the whole attention path on tensors in
// pinned host memory, with the host<->device copies overlapped with compute.
//
// Every (batch, kv head) pair is an independent problem: its G = H / Hkv query
// heads read only that kv head's K and V, the smooth-K mean is per pair, and
// the quantiser and attention kernels work per head.  The problem is cut into
// chunks of consecutive pairs (all G query heads of each); in BHLD layout a
// chunk's Q, K, V and O are contiguous ranges, so a chunk is itself a problem
// with B = 1, H = n * G, Hkv = n.  Chunk c uses device slot c % 3 of the
// caller's workspace:
//   copy-in stream : Q, K, V of chunk c  host -> slot        (after chunk c-3's compute)
//   caller's stream: sa_quantize + attention on the slot      (after its copy-in and
//                                                              chunk c-3's copy-out)
//   copy-out stream: O of chunk c  slot -> host              (after its compute)
// so the copies of one chunk run beside the compute of its neighbours.  The
// host link is the bound (the copies of the whole problem take longer than
// its compute); what no copy-in overlaps is the compute and copy-out of the
// last chunk.  So with the library's chunking of the NVFP4 path the last
// chunks shrink (..., n, n/2, n/4, ...) and a chunk whose attention CTAs
// would leave at least half of the SMs idle runs with split-KV (shares of 8
// key tiles or more, one workspace region that the chunks take in turn on the
// caller's stream).  The kernels compute every head as on the whole problem:
// without split-KV the results are bit-identical to sa_quantize +
// sa_attn_fwd on device buffers; a split NVFP4 chunk differs from them only
// in float32 summation order, as its P is quantised per key tile whatever the
// running maximum.  (The BF16 path rounds P relative to the running maximum,
// which split-KV changes, so its chunks are never split.)

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>
#include <vector>

#include "host_plan.h"
#include "internal.h"

namespace sa {
namespace {

constexpr int kSlots = 3;

// Two copy streams and the events that order the slots, per device; created
// on first use and kept for the life of the process.
struct HostPipe {
  bool ready = false;
  cudaStream_t cin = nullptr, cout = nullptr;
  cudaEvent_t start = nullptr, in[kSlots] = {}, comp[kSlots] = {}, out[kSlots] = {};
  // join: the end of each copy stream's work of a call, for the caller's
  // stream to wait on; last_comp: the last compute of a call on the caller's
  // stream (an overlapped call's compute, and so its use of the split-KV
  // region that all slots share, starts after it)
  cudaEvent_t join_in = nullptr, join_out = nullptr, last_comp = nullptr;
  // the slots of the last call (its workspace and slot size): the slot events
  // order a call after the previous one only when both cut the same memory
  // into the same slots
  const void* last_ws = nullptr;
  size_t last_slot_bytes = 0;
};
HostPipe g_pipe[kMaxDevices];
std::mutex g_pipe_mu;

HostPipe* pipe_for_current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_pipe_mu);
  HostPipe& p = g_pipe[dev];
  if (!p.ready) {
    const unsigned ef = cudaEventDisableTiming;
    if (cudaStreamCreateWithFlags(&p.cin, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&p.cout, cudaStreamNonBlocking) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.start, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.join_in, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.join_out, ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&p.last_comp, ef) != cudaSuccess)
      return nullptr;
    for (int i = 0; i < kSlots; ++i)
      if (cudaEventCreateWithFlags(&p.in[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.comp[i], ef) != cudaSuccess ||
          cudaEventCreateWithFlags(&p.out[i], ef) != cudaSuccess)
        return nullptr;
    p.ready = true;
  }
  return &p;
}

size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

// Byte layout of one slot for chunks of up to n pairs.
struct SlotLayout {
  size_t q, k, v, o, blob, bytes;
};

// The workspace: kSlots slots for the largest chunk, then the split-KV region
// (the largest any chunk needs).
struct PipeLayout {
  SlotLayout slot;
  size_t split, split_bytes, bytes;
};
SlotLayout slot_layout(int n, int G, int L, int d, bool fp4, size_t osz) {
  SlotLayout s;
  const size_t rows_q = (size_t)n * G * L, rows_k = (size_t)n * L;
  size_t off = 0;
  s.q = off, off = al256(off + rows_q * d * 2);
  s.k = off, off = al256(off + rows_k * d * 2);
  s.v = off, off = al256(off + rows_k * d * 2);
  s.o = off, off = al256(off + rows_q * d * osz);
  s.blob = off;
  if (fp4) off = al256(off + sa_fp4_qkv_bytes(1, n * G, n, L, d, nullptr));
  s.bytes = off;
  return s;
}

PipeLayout pipe_layout(const std::vector<Chunk>& plan, int G, int L, int d, bool fp4, size_t osz) {
  int nmax = 0;
  size_t split = 0;
  for (const Chunk& c : plan) {
    nmax = c.n > nmax ? c.n : nmax;
    if (c.nsplit > 1) {
      const size_t b = splitkv_workspace_bytes(Dims{1, c.n * G, c.n, L, L, d}, c.nsplit);
      split = b > split ? b : split;
    }
  }
  PipeLayout p;
  p.slot = slot_layout(nmax, G, L, d, fp4, osz);
  p.split = kSlots * p.slot.bytes;
  p.split_bytes = split;
  p.bytes = p.split + al256(split);
  return p;
}

bool pinned_host(const void* p) {
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeHost;
}

// SA_OK for a problem the pipeline takes (empty ones included: B == 0 or
// L == 0), or the error to return.
sa_status check_host_args(int B, int H, int Hkv, int L, int d, int causal, int mode_flags, int chunk_pairs) {
  if (B < 0 || H <= 0 || Hkv <= 0 || L < 0 || d <= 0 || H % Hkv != 0) return SA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
  if (mode_flags & ~(0xF | SA_OUT_FP32 | SA_HOST_OVERLAP)) return SA_ERR_INVALID_ARG;
  const int mode = mode_flags & 0xF;
  if (mode == SA_MODE_NVFP4_SQ || mode == SA_MODE_NVFP4_FQ) return SA_ERR_UNSUPPORTED;
  if (mode != SA_MODE_BF16 && mode != SA_MODE_NVFP4) return SA_ERR_INVALID_ARG;
  if (chunk_pairs < 0) return SA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return SA_ERR_UNSUPPORTED;
  // a non-empty problem must be one the device calls accept
  if (B > 0 && L > 0 && sa_fp4_qkv_bytes(B, H, Hkv, L, d, nullptr) == 0) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" {

size_t sa_attn_fwd_host_workspace_bytes(int B, int H, int Hkv, int L, int d, int mode_flags, int chunk_pairs) {
  if (check_host_args(B, H, Hkv, L, d, 0, mode_flags, chunk_pairs) != SA_OK || B == 0 || L == 0) return 0;
  const bool fp4 = (mode_flags & 0xF) == SA_MODE_NVFP4;
  const size_t osz = (mode_flags & SA_OUT_FP32) ? 4 : 2;
  return pipe_layout(chunk_plan(B, H, Hkv, L, chunk_pairs, fp4, device_sm_count()), H / Hkv, L, d, fp4, osz).bytes;
}

sa_status sa_attn_fwd_host(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int L, int d,
                           int causal, int mode_flags, void* workspace, size_t workspace_bytes, int chunk_pairs,
                           sa_stream_t stream) {
  sa_status st = check_host_args(B, H, Hkv, L, d, causal, mode_flags, chunk_pairs);
  if (st != SA_OK) return st;
  if (B == 0 || L == 0) return SA_OK;                  // nothing to compute or copy
  if (!q || !k || !v || !o || !workspace) return SA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return SA_ERR_INVALID_ARG;
  if (!pinned_host(q) || !pinned_host(k) || !pinned_host(v) || !pinned_host(o)) return SA_ERR_INVALID_ARG;
  const int G = H / Hkv;
  const bool fp4 = (mode_flags & 0xF) == SA_MODE_NVFP4;
  const std::vector<Chunk> plan = chunk_plan(B, H, Hkv, L, chunk_pairs, fp4, device_sm_count());
  const size_t osz = (mode_flags & SA_OUT_FP32) ? 4 : 2;
  const PipeLayout lay = pipe_layout(plan, G, L, d, fp4, osz);
  if (workspace_bytes < lay.bytes) return SA_ERR_INVALID_ARG;
  HostPipe* p = pipe_for_current_device();
  if (!p) return SA_ERR_CUDA;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const size_t q_pair = (size_t)G * L * d * 2, kv_pair = (size_t)L * d * 2, o_pair = (size_t)G * L * d * osz;
  const uint8_t* hq = static_cast<const uint8_t*>(q);
  const uint8_t* hk = static_cast<const uint8_t*>(k);
  const uint8_t* hv = static_cast<const uint8_t*>(v);
  uint8_t* ho = static_cast<uint8_t*>(o);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  uint8_t* split_ws = ws + lay.split;
  bool ok = true;
  auto cu = [&ok](cudaError_t e) { ok = ok && e == cudaSuccess; };
  // Every exit after the first enqueue makes the caller's stream wait for all
  // the work this call put on the two copy streams, so that synchronising the
  // stream means every copy has finished -- also after an error (the copies
  // already enqueued still read q, k, v and write o and the workspace).
  auto join = [&]() {
    bool j = cudaEventRecord(p->join_in, p->cin) == cudaSuccess;
    j = cudaEventRecord(p->join_out, p->cout) == cudaSuccess && j;
    j = cudaStreamWaitEvent(s, p->join_in, 0) == cudaSuccess && j;
    j = cudaStreamWaitEvent(s, p->join_out, 0) == cudaSuccess && j;
    return j;
  };

  // Both copy streams start after the work already on the caller's stream
  // (an earlier call on the same workspace, for one) -- with SA_HOST_OVERLAP
  // the copy-in stream does not: the first kSlots chunks wait instead for the
  // slot events of the previous call on this device, like later chunks for
  // those of this call (an event never recorded is no wait).  That is only
  // sound when the previous call used the same slots (same workspace, same
  // slot size); otherwise this call waits for everything before it.
  const bool overlap = (mode_flags & SA_HOST_OVERLAP) != 0 && p->last_ws == workspace &&
                       p->last_slot_bytes == lay.slot.bytes;
  // until this call has enqueued all of its work, the next one must not rely
  // on its slot events (an error below returns with the record cleared)
  p->last_ws = nullptr;
  const int dev_mode = mode_flags & ~SA_HOST_OVERLAP;   // the mode of the device-buffer calls
  cu(cudaEventRecord(p->start, s));
  if (!overlap) cu(cudaStreamWaitEvent(p->cin, p->start, 0));
  cu(cudaStreamWaitEvent(p->cout, p->start, 0));
  // an overlapped call may be on another stream than the previous one: its
  // compute waits for the previous call's (the split-KV region is shared by
  // all slots; the slot events cover the rest)
  if (overlap) cu(cudaStreamWaitEvent(s, p->last_comp, 0));
  const int nchunks = (int)plan.size();
  size_t p0 = 0;
  for (int c = 0; ok && c < nchunks; ++c) {
    const int slot = c % kSlots, nc = plan[c].n, nsplit = plan[c].nsplit;
    uint8_t* base = ws + slot * lay.slot.bytes;
    uint8_t *dq = base + lay.slot.q, *dk = base + lay.slot.k, *dv = base + lay.slot.v, *dout = base + lay.slot.o;
    // copy in, once chunk c-3 (or the previous call's last chunk in this
    // slot) is done reading this slot
    if (c >= kSlots || overlap) cu(cudaStreamWaitEvent(p->cin, p->comp[slot], 0));
    cu(cudaMemcpyAsync(dq, hq + p0 * q_pair, nc * q_pair, cudaMemcpyHostToDevice, p->cin));
    cu(cudaMemcpyAsync(dk, hk + p0 * kv_pair, nc * kv_pair, cudaMemcpyHostToDevice, p->cin));
    cu(cudaMemcpyAsync(dv, hv + p0 * kv_pair, nc * kv_pair, cudaMemcpyHostToDevice, p->cin));
    cu(cudaEventRecord(p->in[slot], p->cin));
    // compute, once the inputs are in and chunk c-3's O has left the slot
    cu(cudaStreamWaitEvent(s, p->in[slot], 0));
    if (c >= kSlots || overlap) cu(cudaStreamWaitEvent(s, p->out[slot], 0));
    if (!ok) break;
    const void* aq = dq;
    const void* ak = dk;
    const void* av = dv;
    sa_fp4_qkv x;
    if (fp4) {
      st = sa_fp4_qkv_from_blob(base + lay.slot.blob, 1, nc * G, nc, L, d, &x);
      if (st == SA_OK) st = sa_quantize(dq, dk, dv, 1, nc * G, nc, L, d, &x, stream);
      aq = &x;
      ak = av = nullptr;
    }
    if (st == SA_OK)
      st = nsplit > 1 ? sa_attn_fwd_ws(aq, ak, av, dout, 1, nc * G, nc, L, d, causal, dev_mode, nsplit, split_ws,
                                       lay.split_bytes, stream)
                      : sa_attn_fwd(aq, ak, av, dout, 1, nc * G, nc, L, d, causal, dev_mode, stream);
    if (st != SA_OK) {
      join();
      return st;
    }
    cu(cudaEventRecord(p->comp[slot], s));
    // copy out
    cu(cudaStreamWaitEvent(p->cout, p->comp[slot], 0));
    cu(cudaMemcpyAsync(ho + p0 * o_pair, dout, nc * o_pair, cudaMemcpyDeviceToHost, p->cout));
    cu(cudaEventRecord(p->out[slot], p->cout));
    p0 += nc;
  }
  // the caller's stream completes after the last copy out (and after every
  // copy this call enqueued, also when a step above failed)
  cu(cudaEventRecord(p->last_comp, s));
  const bool joined = join();
  if (!ok || !joined) return SA_ERR_CUDA;
  p->last_ws = workspace;
  p->last_slot_bytes = lay.slot.bytes;
  return SA_OK;
}

}  // extern "C"
