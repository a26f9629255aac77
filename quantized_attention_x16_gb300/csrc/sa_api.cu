// sa_api.cu -- the C ABI declared in include/sa.h: argument validation, TMA
// descriptor encoding, kernel launches on the caller's stream, status codes.
// Nothing here allocates device memory.

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "internal.h"
#include "sm100.cuh"
#include "work.cuh"

namespace sa {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  }
  return fn;
}

// 2-D row-major tensor [outer][inner] of `elem` bytes per element.
bool make_map(CUtensorMap* m, CUtensorMapDataType dt, const void* base, uint64_t inner, uint64_t outer,
              uint32_t elem, uint32_t box_inner, uint32_t box_outer, CUtensorMapSwizzle swz) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * elem};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return fn(m, dt, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// bf16 [B][heads][L][d] (or BLHD) as a 4-D map (channel, token, head, batch)
// with boxes of 64 channels x 128 tokens x 1 x 1, 128B swizzle (the tiles of
// the BF16 attention kernel and the quantiser): a tile that runs past the
// head's last token reads zeros there instead of another head's rows.
bool make_bf16_head_map(CUtensorMap* m, const void* base, int heads, int L, const Dims& dm, bool blhd) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const Strides st = layout_strides(blhd, heads, L, dm.d);
  const cuuint64_t dims[4] = {(cuuint64_t)dm.d, (cuuint64_t)L, (cuuint64_t)heads, (cuuint64_t)dm.B};
  const cuuint64_t strides[3] = {(cuuint64_t)st.t * 2, (cuuint64_t)st.h * 2, (cuuint64_t)st.b * 2};
  const cuuint32_t box[4] = {64, 128, 1, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_bf16_maps(const void* q, const void* k, const void* v, const Dims& dm, bool blhd, CUtensorMap* tq,
                    CUtensorMap* tk, CUtensorMap* tv) {
  return make_bf16_head_map(tq, q, dm.H, dm.Lq, dm, blhd) && make_bf16_head_map(tk, k, dm.Hkv, dm.Lkv, dm, blhd) &&
         make_bf16_head_map(tv, v, dm.Hkv, dm.Lkv, dm, blhd);
}

// SA_OK for sizes the kernels take, or the error to return.  B == 0 or Lq ==
// 0 passes (an empty problem: the entry points return before touching any
// pointer); otherwise Lkv must be positive.
sa_status check_dims(const Dims& dm) {
  if (dm.B < 0 || dm.H <= 0 || dm.Hkv <= 0 || dm.Lq < 0 || dm.Lkv < 0 || dm.d <= 0) return SA_ERR_INVALID_ARG;
  if (dm.H % dm.Hkv != 0) return SA_ERR_INVALID_ARG;
  if (dm.d != 64 && dm.d != 128) return SA_ERR_UNSUPPORTED;
  if (dm.B > 0 && dm.Lq > 0 && dm.Lkv == 0) return SA_ERR_INVALID_ARG;   // queries without keys
  // TMA coordinates are 32-bit: every row index of the padded layouts (and
  // d * B * Hkv) must fit.
  const long long Lqp = ((long long)dm.Lq + 127) / 128 * 128, Lkvp = ((long long)dm.Lkv + 127) / 128 * 128;
  if ((long long)dm.B * dm.H * Lqp >= (1ll << 31) || (long long)dm.B * dm.Hkv * Lkvp >= (1ll << 31) ||
      (long long)dm.B * dm.Hkv * dm.d >= (1ll << 31))
    return SA_ERR_UNSUPPORTED;
  if (dm.H > 65535 || dm.B > 65535) return SA_ERR_UNSUPPORTED;
  return SA_OK;
}

bool empty_problem(const Dims& dm) { return dm.B == 0 || dm.Lq == 0; }

Dims dims_of(const sa_shape* s) { return Dims{s->B, s->H, s->Hkv, s->Lq, s->Lkv, s->d}; }

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Every quantised layout has its length rounded up to 128 token rows.
void blob_sizes(const Dims& dm, size_t sz[8]) {
  const int Lqp = padded_len(dm.Lq), Lkvp = padded_len(dm.Lkv);
  const size_t nq = (size_t)dm.B * dm.H * Lqp, nk = (size_t)dm.B * dm.Hkv * Lkvp;
  const int d = dm.d;
  sz[0] = nq * (d / 2);                                        // q_codes
  sz[1] = (size_t)dm.B * dm.H * (Lqp / 128) * (d / 64) * 512;  // q_sf
  sz[2] = nk * (d / 2);                                        // k_codes
  sz[3] = (size_t)dm.B * dm.Hkv * (Lkvp / 128) * (d / 64) * 512;
  sz[4] = nk * (d / 2);                                        // v_codes (transposed)
  sz[5] = (size_t)dm.B * dm.Hkv * (Lkvp / 64) * 512;           // v_sf
  sz[6] = (size_t)dm.B * dm.Hkv * d * sizeof(float);           // k_mean
  sz[7] = kmean_partial_floats(dm) * sizeof(float);   // K-mean partial sums
}

__global__ void wait_selftest_kernel(uint64_t limit_ns) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);   // expects one arrival that never comes
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(&bar, 0, reinterpret_cast<volatile int*>(&abort_flag), limit_ns);
  __syncthreads();
}

}  // namespace
}  // namespace sa

using namespace sa;

extern "C" {

const char* sa_version(void) { return "sa-gb300 0.1 (sm_103a)"; }

const char* sa_status_string(sa_status s) {
  switch (s) {
    case SA_OK: return "ok";
    case SA_ERR_INVALID_ARG: return "invalid argument";
    case SA_ERR_UNSUPPORTED: return "unsupported size";
    case SA_ERR_CUDA: return "CUDA error";
    case SA_ERR_TIMEOUT: return "device barrier wait timed out";
  }
  return "unknown status";
}

size_t sa_fp4_qkv_bytes_s(const sa_shape* shape, size_t offsets_out[8]) {
  if (!shape) return 0;
  const Dims dm = dims_of(shape);
  if (check_dims(dm) != SA_OK || dm.B == 0 || dm.Lq == 0 || dm.Lkv == 0) return 0;
  size_t sz[8];
  blob_sizes(dm, sz);
  size_t off = 0;
  for (int i = 0; i < 8; ++i) {
    if (offsets_out) offsets_out[i] = off;
    off = align256(off + sz[i]);
  }
  return off;
}

size_t sa_fp4_qkv_bytes(int B, int H, int Hkv, int L, int d, size_t offsets_out[8]) {
  const sa_shape s{B, H, Hkv, L, L, d};
  return sa_fp4_qkv_bytes_s(&s, offsets_out);
}

sa_status sa_fp4_qkv_from_blob_s(void* blob, const sa_shape* shape, sa_fp4_qkv* out) {
  if (!out || !blob || !shape || (reinterpret_cast<uintptr_t>(blob) & 255u)) return SA_ERR_INVALID_ARG;
  size_t off[8];
  if (sa_fp4_qkv_bytes_s(shape, off) == 0) {
    const sa_status st = check_dims(dims_of(shape));
    return st != SA_OK ? st : SA_ERR_INVALID_ARG;     // an empty problem has no blob
  }
  uint8_t* p = static_cast<uint8_t*>(blob);
  out->q_codes = p + off[0];
  out->q_sf = p + off[1];
  out->k_codes = p + off[2];
  out->k_sf = p + off[3];
  out->v_codes = p + off[4];
  out->v_sf = p + off[5];
  out->k_mean = reinterpret_cast<float*>(p + off[6]);
  out->workspace = p + off[7];
  return SA_OK;
}

sa_status sa_fp4_qkv_from_blob(void* blob, int B, int H, int Hkv, int L, int d, sa_fp4_qkv* out) {
  const sa_shape s{B, H, Hkv, L, L, d};
  return sa_fp4_qkv_from_blob_s(blob, &s, out);
}

static bool fp4_ptrs_ok(const sa_fp4_qkv* x) {
  return x && aligned16(x->q_codes) && aligned16(x->q_sf) && aligned16(x->k_codes) && aligned16(x->k_sf) &&
         aligned16(x->v_codes) && aligned16(x->v_sf) && aligned16(x->k_mean) && aligned16(x->workspace);
}

sa_status sa_quantize_s(const void* q, const void* k, const void* v, const sa_shape* shape, int flags,
                        const sa_fp4_qkv* out, sa_stream_t stream) {
  if (!shape) return SA_ERR_INVALID_ARG;
  const Dims dm = dims_of(shape);
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (flags & ~SA_LAYOUT_BLHD) return SA_ERR_INVALID_ARG;
  if (dm.B == 0 || (dm.Lq == 0 && dm.Lkv == 0)) return SA_OK;
  if (dm.Lq == 0) return SA_ERR_INVALID_ARG;            // keys without queries: nothing to quantise them for
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !fp4_ptrs_ok(out)) return SA_ERR_INVALID_ARG;
  const bool blhd = (flags & SA_LAYOUT_BLHD) != 0;
  CUtensorMap tq, tk, tv;
  if (!make_bf16_maps(q, k, v, dm, blhd, &tq, &tk, &tv)) return SA_ERR_CUDA;
  return launch_quantize(dm, *out, tq, tk, tv, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

sa_status sa_quantize_kv_s(const void* k, const void* v, const sa_shape* shape, int flags, const sa_fp4_qkv* out,
                           sa_stream_t stream) {
  if (!shape) return SA_ERR_INVALID_ARG;
  const Dims dm = dims_of(shape);
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (flags & ~SA_LAYOUT_BLHD) return SA_ERR_INVALID_ARG;
  if (dm.B == 0 || (dm.Lq == 0 && dm.Lkv == 0)) return SA_OK;
  if (dm.Lq == 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !out || !aligned16(out->k_codes) || !aligned16(out->k_sf) ||
      !aligned16(out->v_codes) || !aligned16(out->v_sf) || !aligned16(out->k_mean) || !aligned16(out->workspace))
    return SA_ERR_INVALID_ARG;
  const bool blhd = (flags & SA_LAYOUT_BLHD) != 0;
  CUtensorMap tk, tv;
  if (!make_bf16_head_map(&tk, k, dm.Hkv, dm.Lkv, dm, blhd) || !make_bf16_head_map(&tv, v, dm.Hkv, dm.Lkv, dm, blhd))
    return SA_ERR_CUDA;
  // (the Q map is not read: pass 1 takes the K-mean tiles only)
  return launch_quantize(dm, *out, tk, tk, tv, reinterpret_cast<cudaStream_t>(stream), false) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

sa_status sa_quantize_ex(const void* q, const void* k, const void* v, int B, int H, int Hkv, int L, int d, int flags,
                         const sa_fp4_qkv* out, sa_stream_t stream) {
  const sa_shape s{B, H, Hkv, L, L, d};
  return sa_quantize_s(q, k, v, &s, flags, out, stream);
}

sa_status sa_quantize(const void* q, const void* k, const void* v, int B, int H, int Hkv, int L, int d,
                      const sa_fp4_qkv* out, sa_stream_t stream) {
  const sa_shape s{B, H, Hkv, L, L, d};
  return sa_quantize_s(q, k, v, &s, 0, out, stream);
}

sa_status sa_quantize_static_scratch(const void* q, const void* k, const void* v, int B, int H, int Hkv, int L,
                                     int d, const sa_fp4_qkv* out, sa_stream_t stream) {
  const Dims dm{B, H, Hkv, L, L, d};
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (empty_problem(dm)) return SA_OK;
  if (kmean_partial_floats(dm) > kStaticScratchFloats) return SA_ERR_UNSUPPORTED;   // before any pointer check
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !out || !aligned16(out->q_codes) ||
      !aligned16(out->q_sf) || !aligned16(out->k_codes) || !aligned16(out->k_sf) || !aligned16(out->v_codes) ||
      !aligned16(out->v_sf) || !aligned16(out->k_mean))
    return SA_ERR_INVALID_ARG;
  CUtensorMap tq, tk, tv;
  if (!make_bf16_maps(q, k, v, dm, false, &tq, &tk, &tv)) return SA_ERR_CUDA;
  return launch_quantize_static_scratch(dm, *out, tq, tk, tv, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

static void smooth_q_sizes(const Dims& dm, size_t sz[2]) {
  const size_t tiles = (size_t)dm.B * dm.H * (padded_len(dm.Lq) / 128);
  sz[0] = tiles * dm.d * sizeof(float);                         // q_mean
  sz[1] = tiles * padded_len(dm.Lkv) * sizeof(float);           // ds
}

size_t sa_smooth_q_bytes_s(const sa_shape* shape, size_t offsets_out[2]) {
  if (!shape) return 0;
  const Dims dm = dims_of(shape);
  if (check_dims(dm) != SA_OK || dm.B == 0 || dm.Lq == 0 || dm.Lkv == 0) return 0;
  size_t sz[2];
  smooth_q_sizes(dm, sz);
  if (offsets_out) {
    offsets_out[0] = 0;
    offsets_out[1] = align256(sz[0]);
  }
  return align256(align256(sz[0]) + sz[1]);
}

sa_status sa_smooth_q_from_blob_s(void* blob, const sa_shape* shape, sa_fp4_sq* out) {
  if (!out || !blob || !shape || (reinterpret_cast<uintptr_t>(blob) & 255u)) return SA_ERR_INVALID_ARG;
  size_t off[2];
  if (sa_smooth_q_bytes_s(shape, off) == 0) {
    const sa_status st = check_dims(dims_of(shape));
    return st != SA_OK ? st : SA_ERR_INVALID_ARG;
  }
  uint8_t* p = static_cast<uint8_t*>(blob);
  out->q_mean = reinterpret_cast<float*>(p + off[0]);
  out->ds = reinterpret_cast<float*>(p + off[1]);
  return SA_OK;
}

sa_status sa_quantize_smooth_q(const void* q, const sa_shape* shape, int flags, const sa_fp4_sq* x,
                               sa_stream_t stream) {
  if (!shape || !x) return SA_ERR_INVALID_ARG;
  const Dims dm = dims_of(shape);
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (flags & ~SA_LAYOUT_BLHD) return SA_ERR_INVALID_ARG;
  if (empty_problem(dm)) return SA_OK;
  if (dm.Lkv == 0) return SA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(x->fp4.q_codes) || !aligned16(x->fp4.q_sf) || !aligned16(x->fp4.k_codes) ||
      !aligned16(x->fp4.k_sf) || !aligned16(x->q_mean) || !aligned16(x->ds))
    return SA_ERR_INVALID_ARG;
  const Strides sq = layout_strides((flags & SA_LAYOUT_BLHD) != 0, dm.H, dm.Lq, dm.d);
  return launch_smooth_q(q, sq, dm, x->fp4, x->q_mean, x->ds, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

// The work split: `requested` 0 = the library's choice, 1 = one unit per CTA,
// n > 1 = split-KV with n shares (at most one per key tile), -1 = stream-K.
// The library chooses stream-K for the NVFP4 path when the pairs alone can
// fill every SM (measured on one GB300 in one process, llm_prefill NVFP4
// attention: 198.7 us for one pair per CTA before the persistent form, 196.6
// us one pair per CTA now, 194.5 us stream-K, operands L2-resident after the
// quantiser; 201.4 / 197.3 / 195.2 us after an L2 flush), split-KV when the
// pairs leave half of the SMs idle and the shares stay long, else one unit
// per CTA.
// NVFP4 calls that run on the few-row decode kernel (the smooth-Q variant
// always runs on the prefill kernel).
static bool use_decode(const Dims& dm, int mode) { return mode == SA_MODE_NVFP4 && decode_eligible(dm); }
static bool is_fp4(int mode) {
  return mode == SA_MODE_NVFP4 || mode == SA_MODE_NVFP4_SQ || mode == SA_MODE_NVFP4_FQ;
}

static int resolve_nsplit(const Dims& dm, int causal, int mode, int requested) {
  if (requested == 1) return 1;
  if (requested == kStreamK) return kStreamK;
  const int sms = device_sm_count();
  // few query rows per kv head (decode): the decode kernel, its key range cut
  // into shares so that the (batch, kv head) pairs fill one wave of CTAs
  // (equal ranges of (pair, key tile) items, kStreamK, measured slower:
  // decode_gqa 60 against 45.6 us)
  if (requested == 0 && use_decode(dm, mode)) return decode_nsplit(dm, sms);
  if (requested == 0) {
    const long long pairs = (long long)(((dm.Lq + 127) / 128 + 1) / 2) * dm.B * dm.H;
    // stream-K balances key tiles, not units: under the causal mask most
    // pairs are short, the per-unit fixed cost (~6 us) dominates the ranges
    // that hold them, and the heaviest-first work list is faster (causal GQA
    // B1 H32 L8192: 366 us against 533 us)
    if (is_fp4(mode) && !causal && sms > 0 && pairs >= sms &&
        streamk_fits(dm.B, dm.H, dm.Lq, dm.Lkv, causal))
      return kStreamK;
    return choose_nsplit(dm.B, dm.H, dm.Lq, dm.Lkv, sms);
  }
  const int nkt = (dm.Lkv + 127) / 128;
  return requested < nkt ? requested : nkt;
}

static size_t work_split_bytes(const Dims& dm, int causal, int mode, int nsplit) {
  // (kStreamK is an NVFP4 schedule; for decode shapes, the decode kernel's ranges)
  if (nsplit == kStreamK && use_decode(dm, mode)) return decode_range_workspace_bytes(dm, device_sm_count());
  if (nsplit == kStreamK) {
    int ctas = 0;
    make_streamk_work(dm.B, dm.H, dm.Lq, dm.Lkv, causal, device_sm_count() > 0 ? device_sm_count() : 1, &ctas);
    return streamk_workspace_bytes(dm, ctas);
  }
  return splitkv_workspace_bytes(dm, nsplit);
}

static sa_status attn_fwd_impl(const void* q, const void* k, const void* v, void* o, const Dims& dm, int causal,
                               int mode_flags, int nsplit_req, void* workspace, size_t workspace_bytes,
                               sa_stream_t stream) {
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (causal != 0 && causal != 1) return SA_ERR_INVALID_ARG;
  if (causal && dm.Lkv < dm.Lq) return SA_ERR_INVALID_ARG;   // the first queries would see no key
  if (mode_flags & ~(0xF | SA_OUT_FP32 | SA_LAYOUT_BLHD)) return SA_ERR_INVALID_ARG;
  const int mode = mode_flags & 0xF;
  if (mode != SA_MODE_BF16 && !is_fp4(mode)) return SA_ERR_INVALID_ARG;
  if (nsplit_req < kStreamK) return SA_ERR_INVALID_ARG;
  if (nsplit_req == kStreamK &&
      (!is_fp4(mode) || (!use_decode(dm, mode) && !streamk_fits(dm.B, dm.H, dm.Lq, dm.Lkv, causal))))
    return SA_ERR_UNSUPPORTED;
  if (empty_problem(dm)) return SA_OK;
  const bool out_f32 = (mode_flags & SA_OUT_FP32) != 0;
  const bool blhd = (mode_flags & SA_LAYOUT_BLHD) != 0;
  if (!aligned16(o)) return SA_ERR_INVALID_ARG;
  const Strides so = layout_strides(blhd, dm.H, dm.Lq, dm.d);            // O strides
  // split-KV and stream-K only with a workspace large enough for the partial
  // results (a forced choice without one is an argument error; the library's
  // own choice then falls back to one unit per CTA)
  int nsplit = resolve_nsplit(dm, causal, mode, nsplit_req);
  const bool needs_ws = nsplit > 1 || nsplit == kStreamK;
  const bool ws_ok = workspace != nullptr && workspace_bytes >= work_split_bytes(dm, causal, mode, nsplit);
  if (needs_ws && !ws_ok && nsplit_req != 0) return SA_ERR_INVALID_ARG;
  if (needs_ws && !ws_ok) nsplit = 1;
  if (nsplit != 1 && !aligned16(workspace)) return SA_ERR_INVALID_ARG;
  SplitOut part{nullptr, nullptr};
  if (nsplit > 1) part = splitkv_layout(workspace, dm, nsplit);
  if (nsplit == kStreamK && use_decode(dm, mode)) {
    part = decode_range_layout(workspace, dm, device_sm_count());
  } else if (nsplit == kStreamK) {
    int ctas = 0;
    make_streamk_work(dm.B, dm.H, dm.Lq, dm.Lkv, causal, device_sm_count() > 0 ? device_sm_count() : 1, &ctas);
    part = streamk_layout(workspace, dm, ctas);
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  CUtensorMap tq, tk, tv;
  if (mode == SA_MODE_BF16) {
    if (!aligned16(q) || !aligned16(k) || !aligned16(v)) return SA_ERR_INVALID_ARG;
    if (!make_bf16_head_map(&tq, q, dm.H, dm.Lq, dm, blhd) || !make_bf16_head_map(&tk, k, dm.Hkv, dm.Lkv, dm, blhd) ||
        !make_bf16_head_map(&tv, v, dm.Hkv, dm.Lkv, dm, blhd))
      return SA_ERR_CUDA;
    return launch_attn_bf16(tq, tk, tv, o, so, dm, causal, out_f32, nsplit, part, s) == cudaSuccess ? SA_OK
                                                                                                    : SA_ERR_CUDA;
  }
  // SA_MODE_NVFP4_FQ: q is the bf16 Q, k the sa_fp4_qkv of K and V (its Q
  // buffers unused); otherwise q is the sa_fp4_qkv (SA_MODE_NVFP4) or the
  // sa_fp4_sq, whose first member is the sa_fp4_qkv (SA_MODE_NVFP4_SQ)
  const bool fq = mode == SA_MODE_NVFP4_FQ;
  if (fq ? (q == nullptr || k == nullptr || v != nullptr || !aligned16(q))
         : (k != nullptr || v != nullptr || q == nullptr))
    return SA_ERR_INVALID_ARG;
  const sa_fp4_sq* xs = mode == SA_MODE_NVFP4_SQ ? static_cast<const sa_fp4_sq*>(q) : nullptr;
  const sa_fp4_qkv* x = fq ? static_cast<const sa_fp4_qkv*>(k) : (xs ? &xs->fp4 : static_cast<const sa_fp4_qkv*>(q));
  if (xs && !aligned16(xs->ds)) return SA_ERR_INVALID_ARG;
  if ((!fq && (!aligned16(x->q_codes) || !aligned16(x->q_sf))) || !aligned16(x->k_codes) || !aligned16(x->k_sf) ||
      !aligned16(x->v_codes) || !aligned16(x->v_sf))
    return SA_ERR_INVALID_ARG;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int d = dm.d;
  const CUtensorMapSwizzle qk_swz = d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  // the quantised layouts hold whole 128-token tiles
  const int Lqp = padded_len(dm.Lq), Lkvp = padded_len(dm.Lkv);
  if (!(fq ? make_bf16_head_map(&tq, q, dm.H, dm.Lq, dm, blhd)
           : make_map(&tq, u8, x->q_codes, d / 2, (uint64_t)dm.B * dm.H * Lqp, 1, d / 2, 128, qk_swz)) ||
      !make_map(&tk, u8, x->k_codes, d / 2, (uint64_t)dm.B * dm.Hkv * Lkvp, 1, d / 2, 128, qk_swz) ||
      !make_map(&tv, u8, x->v_codes, Lkvp / 2, (uint64_t)dm.B * dm.Hkv * d, 1, 64, d, CU_TENSOR_MAP_SWIZZLE_64B))
    return SA_ERR_CUDA;
  // at most 16 query rows per kv head (decode): the decode kernel (stream-K
  // there means its balanced ranges)
  if (use_decode(dm, mode))
    return launch_attn_decode(tk, tv, *x, o, so, dm, causal, out_f32, nsplit, part, s) == cudaSuccess ? SA_OK
                                                                                                      : SA_ERR_CUDA;
  return launch_attn_nvfp4(tq, tk, tv, *x, o, so, dm, causal, out_f32, nsplit, part, s, xs ? xs->ds : nullptr, fq) ==
                 cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

sa_status sa_attn_fwd(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int L, int d,
                      int causal, int mode_flags, sa_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, Dims{B, H, Hkv, L, L, d}, causal, mode_flags, 1, nullptr, 0, stream);
}

size_t sa_attn_fwd_workspace_bytes_s(const sa_shape* shape, int causal, int mode, int nsplit) {
  if (!shape) return 0;
  const Dims dm = dims_of(shape);
  const int m = mode & 0xF;
  if (check_dims(dm) != SA_OK || empty_problem(dm) || nsplit < kStreamK) return 0;
  if (causal != 0 && causal != 1) return 0;
  if (nsplit == kStreamK && !is_fp4(m)) return 0;
  return work_split_bytes(dm, causal, m, resolve_nsplit(dm, causal, m, nsplit));
}

size_t sa_attn_fwd_workspace_bytes(int B, int H, int Hkv, int L, int d, int causal, int mode, int nsplit) {
  const sa_shape s{B, H, Hkv, L, L, d};
  return sa_attn_fwd_workspace_bytes_s(&s, causal, mode, nsplit);
}

sa_status sa_attn_fwd_s(const void* q, const void* k, const void* v, void* o, const sa_shape* shape, int causal,
                        int mode, int nsplit, void* workspace, size_t workspace_bytes, sa_stream_t stream) {
  if (!shape) return SA_ERR_INVALID_ARG;
  return attn_fwd_impl(q, k, v, o, dims_of(shape), causal, mode, nsplit, workspace, workspace_bytes, stream);
}

sa_status sa_attn_fwd_ws(const void* q, const void* k, const void* v, void* o, int B, int H, int Hkv, int L, int d,
                         int causal, int mode, int nsplit, void* workspace, size_t workspace_bytes,
                         sa_stream_t stream) {
  return attn_fwd_impl(q, k, v, o, Dims{B, H, Hkv, L, L, d}, causal, mode, nsplit, workspace, workspace_bytes,
                       stream);
}

sa_status sa_last_device_error(void) {
  int e1 = 0, e2 = 0, e3 = 0, e4 = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return SA_ERR_CUDA;
  if (attn_bf16_read_error(&e1) != cudaSuccess || attn_nvfp4_read_error(&e2) != cudaSuccess ||
      quant_read_error(&e4) != cudaSuccess || read_and_clear_device_error(&e3) != cudaSuccess)
    return SA_ERR_CUDA;
  const int e = e1 ? e1 : (e2 ? e2 : (e4 ? e4 : e3));
  return e ? static_cast<sa_status>(e) : SA_OK;
}

sa_status sa_selftest_nvfp4_score_tile(const sa_fp4_qkv* x, const sa_shape* shape, int b, int h, int qt, int kt,
                                       float* s_out, sa_stream_t stream) {
  if (!shape || !x || !s_out) return SA_ERR_INVALID_ARG;
  const Dims dm = dims_of(shape);
  const sa_status st = check_dims(dm);
  if (st != SA_OK) return st;
  if (empty_problem(dm)) return SA_ERR_INVALID_ARG;                 // no tile to compute
  if (b < 0 || b >= dm.B || h < 0 || h >= dm.H || qt < 0 || qt >= padded_len(dm.Lq) / 128 || kt < 0 ||
      kt >= padded_len(dm.Lkv) / 128)
    return SA_ERR_INVALID_ARG;
  if (!aligned16(x->q_codes) || !aligned16(x->q_sf) || !aligned16(x->k_codes) || !aligned16(x->k_sf) ||
      !aligned16(s_out))
    return SA_ERR_INVALID_ARG;
  const CUtensorMapDataType u8 = CU_TENSOR_MAP_DATA_TYPE_UINT8;
  const int d = dm.d;
  const CUtensorMapSwizzle qk_swz = d == 128 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_32B;
  const int Lqp = padded_len(dm.Lq), Lkvp = padded_len(dm.Lkv);
  CUtensorMap tq, tk;
  if (!make_map(&tq, u8, x->q_codes, d / 2, (uint64_t)dm.B * dm.H * Lqp, 1, d / 2, 128, qk_swz) ||
      !make_map(&tk, u8, x->k_codes, d / 2, (uint64_t)dm.B * dm.Hkv * Lkvp, 1, d / 2, 128, qk_swz))
    return SA_ERR_CUDA;
  return launch_nvfp4_score_tile(tq, tk, *x, dm, b, h, qt, kt, s_out, reinterpret_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

sa_status sa_selftest_exp_path(const float* x, const float* y, int n, float* ex2_out, float* lg2_out,
                                sa_stream_t stream) {
  if (n < 0 || (n > 0 && (!x || !y || !ex2_out || !lg2_out))) return SA_ERR_INVALID_ARG;
  return launch_exp_path_selftest(x, y, n, ex2_out, lg2_out, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? SA_OK
             : SA_ERR_CUDA;
}

sa_status sa_selftest_wait_timeout(uint64_t limit_ns, sa_stream_t stream) {
  if (limit_ns == 0 || limit_ns > 10000000000ull) return SA_ERR_INVALID_ARG;
  wait_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(limit_ns);
  return cudaGetLastError() == cudaSuccess ? SA_OK : SA_ERR_CUDA;
}

}  // extern "C"
