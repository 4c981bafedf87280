// Host layer of libfdma: argument validation, workspace layout, TMA tensor
// maps and kernel launches behind the C ABI declared in include/fdma.h.
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "fdma_internal.h"

namespace fdma {

__device__ int g_device_error;  // first kernel-side error code (0 = none)

namespace {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int* device_error_word() {
  static std::mutex mu;
  static std::unordered_map<int, int*> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int* ptr = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&ptr), g_device_error) != cudaSuccess) return nullptr;
  cache[dev] = ptr;
  return ptr;
}

inline int cdiv(int a, int b) { return (a + b - 1) / b; }
inline size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }
inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int validate(const fdma_args* a, bool need_workspace) {
  if (a == nullptr) return FDMA_ERR_INVALID;
  if (a->B <= 0 || a->Nq <= 0 || a->Nk <= 0 || a->Hq <= 0 || a->Hkv <= 0) return FDMA_ERR_INVALID;
  if (a->Hq % a->Hkv != 0) return FDMA_ERR_INVALID;
  if (a->dv < 0) return FDMA_ERR_INVALID;
  if (!head_dims_ok(a->d, head_dim_v(*a))) return FDMA_ERR_UNSUPPORTED;
  if (cdiv(a->Nk, kTile) > kMaxKTiles || cdiv(a->Nq, kTile) > kMaxKTiles) return FDMA_ERR_UNSUPPORTED;
  if (!(std::isfinite(a->scale) && a->scale > 0.f)) return FDMA_ERR_INVALID;
  if (a->is_causal < 0 || a->is_causal > 2) return FDMA_ERR_INVALID;
  if (a->is_causal == 2 && (a->q_offset > (1 << 30) || a->q_offset < -(1 << 30))) return FDMA_ERR_INVALID;
  if (a->q == nullptr || a->k == nullptr || a->v == nullptr) return FDMA_ERR_INVALID;
  for (const void* p : {a->q, a->k, a->v})
    if (!aligned16(p)) return FDMA_ERR_UNSUPPORTED;
  for (const int64_t* st : {a->q_stride, a->k_stride, a->v_stride})
    for (int i = 0; i < 3; ++i)
      if (st[i] < 0 || (st[i] * 2) % 16 != 0) return FDMA_ERR_UNSUPPORTED;
  switch (a->mask_kind) {
    case FDMA_MASK_NONE:
      break;
    case FDMA_MASK_DENSE:
    case FDMA_MASK_DENSE_U8:
      if (a->mask == nullptr) return FDMA_ERR_INVALID;
      if (!aligned16(a->mask)) return FDMA_ERR_UNSUPPORTED;
      for (int i = 0; i < 3; ++i)  // rows are read in pieces of 8 elements
        if (a->mask_stride[i] < 0 || a->mask_stride[i] % 8 != 0) return FDMA_ERR_UNSUPPORTED;
      break;
    case FDMA_MASK_BITS:
      if (a->mask == nullptr) return FDMA_ERR_INVALID;
      for (int i = 0; i < 3; ++i)
        if (a->mask_stride[i] < 0) return FDMA_ERR_INVALID;
      break;
    case FDMA_MASK_COLRANGES:
    case FDMA_MASK_COLRANGES2:
      if (a->colranges == nullptr) return FDMA_ERR_INVALID;
      if (a->cr_stride[0] < 0 || a->cr_stride[1] < 0) return FDMA_ERR_INVALID;
      break;
    default:
      return FDMA_ERR_INVALID;
  }
  if (a->bias != nullptr) {
    if (!aligned16(a->bias)) return FDMA_ERR_UNSUPPORTED;
    if (a->Nk % 8 != 0) return FDMA_ERR_UNSUPPORTED;
    for (int i = 0; i < 3; ++i)
      if (a->bias_stride[i] < 0 || (a->bias_stride[i] * 2) % 16 != 0) return FDMA_ERR_UNSUPPORTED;
    if (a->bias_stride[2] == 0 && a->Nq > 1) return FDMA_ERR_UNSUPPORTED;  // rows must be distinct
  }
  if (need_workspace && (a->workspace == nullptr || (reinterpret_cast<uintptr_t>(a->workspace) & 255u) != 0))
    return FDMA_ERR_WORKSPACE;
  return FDMA_OK;
}

// 4D bf16 tensor map with a 64 x 128 box (128-byte swizzle): dims listed
// innermost first, strides (bytes) for dims 1..3.  A size-1 dim accepts any stride.
bool make_map(CUtensorMap* m, const void* base, const uint64_t dims[4], const uint64_t strides_b[3]) {
  EncodeTiledFn enc = encode_fn();
  if (enc == nullptr) return false;
  cuuint64_t gd[4] = {dims[0], dims[1], dims[2], dims[3]};
  cuuint64_t gs[3];
  for (int i = 0; i < 3; ++i) {
    uint64_t s = strides_b[i];
    // an extent-1 (unused or broadcast) dim given stride 0 gets the stride of a packed layout
    if (s == 0) s = (i == 0) ? ((dims[0] * 2 + 15) / 16) * 16 : gs[i - 1] * dims[i];
    gs[i] = s;
  }
  cuuint32_t box[4] = {64, 128, 1, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), gd, gs, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Bias (B,Hkv,Nq,Nk) as a 4D map; an axis with stride 0 (broadcast) gets extent 1 and is
// addressed with coordinate 0 by the kernels (bias_bsel / bias_hsel = 0).
bool bias_map(CUtensorMap* m, const fdma_args* a) {
  const bool bb = a->bias_stride[0] == 0, bh = a->bias_stride[1] == 0;
  const uint64_t dims[4] = {static_cast<uint64_t>(a->Nk), static_cast<uint64_t>(a->Nq),
                            bh ? 1ull : static_cast<uint64_t>(a->Hkv), bb ? 1ull : static_cast<uint64_t>(a->B)};
  const uint64_t sb[3] = {static_cast<uint64_t>(a->bias_stride[2]) * 2, static_cast<uint64_t>(a->bias_stride[1]) * 2,
                          static_cast<uint64_t>(a->bias_stride[0]) * 2};
  return make_map(m, a->bias, dims, sb);
}

bool bshd_map(CUtensorMap* m, const void* base, int B, int N, int H, int d, const int64_t st[3]) {
  const uint64_t dims[4] = {static_cast<uint64_t>(d), static_cast<uint64_t>(N), static_cast<uint64_t>(H),
                            static_cast<uint64_t>(B)};
  const uint64_t sb[3] = {static_cast<uint64_t>(st[1]) * 2, static_cast<uint64_t>(st[2]) * 2,
                          static_cast<uint64_t>(st[0]) * 2};
  if ((B > 1 && st[0] == 0) || (H > 1 && st[2] == 0) || (N > 1 && st[1] == 0)) return false;
  return make_map(m, base, dims, sb);
}

int classify_into_workspace(const fdma_args* a, int8_t* user_map, cudaStream_t stream) {
  const WorkspaceLayout w = workspace_layout(a->B, a->Nq, a->Nk, a->Hq, a->Hkv, a->d);
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  ClassifyParams p{};
  p.B = a->B;
  p.Nq = a->Nq;
  p.Nk = a->Nk;
  p.Hkv = a->Hkv;
  p.nTq = cdiv(a->Nq, kTile);
  p.nTk = cdiv(a->Nk, kTile);
  p.mask_kind = a->mask_kind;
  p.causal = a->is_causal ? 1 : 0;
  p.causal_off = a->is_causal == 2 ? a->q_offset : a->Nk - a->Nq;
  p.no_skip = (a->flags & FDMA_FLAG_NO_SKIP) ? 1 : 0;
  p.mask = static_cast<const uint16_t*>(a->mask);
  p.mask_u8 = static_cast<const uint8_t*>(a->mask);
  p.ms_b = a->mask_stride[0];
  p.ms_h = a->mask_stride[1];
  p.ms_r = a->mask_stride[2];
  p.cr = a->colranges;
  p.cr_b = a->cr_stride[0];
  p.cr_h = a->cr_stride[1];
  p.kmap = reinterpret_cast<int8_t*>(ws + w.kmap);
  p.user_map = user_map;
  p.bits_row = reinterpret_cast<uint4*>(ws + w.bits_row);
  p.bits_col = reinterpret_cast<uint4*>(ws + w.bits_col);
  if (a->mask_kind == FDMA_MASK_DENSE && (a->mask_stride[2] > 0 || a->Nq == 1)) {
    // bf16 masks stream through TMA; an axis with stride 0 (broadcast) gets extent 1.  A row
    // stride of 0 (one mask row for every query) or a layout the tensor map refuses takes the
    // register-load kernel below.
    const bool bb = a->mask_stride[0] == 0, bh = a->mask_stride[1] == 0;
    const uint64_t dims[4] = {static_cast<uint64_t>(a->Nk), static_cast<uint64_t>(a->Nq),
                              bh ? 1ull : static_cast<uint64_t>(a->Hkv), bb ? 1ull : static_cast<uint64_t>(a->B)};
    const uint64_t sb[3] = {static_cast<uint64_t>(a->mask_stride[2]) * 2, static_cast<uint64_t>(a->mask_stride[1]) * 2,
                            static_cast<uint64_t>(a->mask_stride[0]) * 2};
    CUtensorMap tm;
    p.err = device_error_word();
    if (p.err == nullptr) return FDMA_ERR_CUDA;
    if (make_map(&tm, a->mask, dims, sb)) {
      p.mask_bsel = bb ? 0 : 1;
      p.mask_hsel = bh ? 0 : 1;
      return launch_classify_tma1(tm, p, stream) == cudaSuccess ? FDMA_OK : FDMA_ERR_CUDA;
    }
  }
  return launch_classify(p, stream) == cudaSuccess ? FDMA_OK : FDMA_ERR_CUDA;
}

}  // namespace

WorkspaceLayout workspace_layout(int B, int Nq, int Nk, int Hq, int Hkv, int d) {
  WorkspaceLayout w{};
  const size_t nTq = static_cast<size_t>(cdiv(Nq, kTile)), nTk = static_cast<size_t>(cdiv(Nk, kTile));
  const size_t tiles = static_cast<size_t>(B) * Hkv * nTq * nTk;
  const size_t nqpad = nTq * kTile;
  size_t off = 0;
  w.kmap = off;
  off = align256(off + tiles);
  w.bits_row = off;
  off = align256(off + tiles * kTile * 16);
  w.bits_col = off;
  off = align256(off + tiles * kTile * 16);
  w.total_fwd = off;
  w.lse2 = off;
  off = align256(off + static_cast<size_t>(B) * Hq * nqpad * 4);
  w.delta = off;
  off = align256(off + static_cast<size_t>(B) * Hq * nqpad * 4);
  w.dq_acc = off;
  off = align256(off + static_cast<size_t>(B) * nqpad * Hq * dq_acc_width(d) * 4);
  w.total_bwd = off;
  return w;
}

}  // namespace fdma

using namespace fdma;

extern "C" {

size_t fdma_workspace_size(const fdma_args* a, int for_bwd) {
  if (a == nullptr || a->B <= 0 || a->Nq <= 0 || a->Nk <= 0 || a->Hq <= 0 || a->Hkv <= 0 || a->Hq % a->Hkv ||
      a->dv < 0 || !head_dims_ok(a->d, head_dim_v(*a)))
    return 0;
  const WorkspaceLayout w = workspace_layout(a->B, a->Nq, a->Nk, a->Hq, a->Hkv, a->d);
  return for_bwd ? w.total_bwd : w.total_fwd;
}

int fdma_classify_blocks(const fdma_args* a, int block_m, int block_n, int8_t* block_map, void* stream) {
  int st = validate(a, true);
  if (st != FDMA_OK) return st;
  if (block_m != kTile || block_n != kTile) return FDMA_ERR_UNSUPPORTED;
  if (a->workspace_bytes < fdma_workspace_size(a, 0)) return FDMA_ERR_WORKSPACE;
  return classify_into_workspace(a, block_map, static_cast<cudaStream_t>(stream));
}

int fdma_fwd(const fdma_args* a, void* out, float* lse, void* stream_v) {
  int st = validate(a, true);
  if (st != FDMA_OK) return st;
  if (out == nullptr || lse == nullptr) return FDMA_ERR_INVALID;
  if (!aligned16(out)) return FDMA_ERR_UNSUPPORTED;
  if (a->workspace_bytes < fdma_workspace_size(a, 0)) return FDMA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int* err = device_error_word();
  if (err == nullptr) return FDMA_ERR_CUDA;
  if (!(a->flags & FDMA_FLAG_REUSE_CLASSIFICATION)) {
    st = classify_into_workspace(a, nullptr, stream);
    if (st != FDMA_OK) return st;
  }
  const WorkspaceLayout w = workspace_layout(a->B, a->Nq, a->Nk, a->Hq, a->Hkv, a->d);
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  CUtensorMap tq, tk, tv, tb;
  const int dv = head_dim_v(*a);
  if (!bshd_map(&tq, a->q, a->B, a->Nq, a->Hq, a->d, a->q_stride) ||
      !bshd_map(&tk, a->k, a->B, a->Nk, a->Hkv, a->d, a->k_stride) ||
      !bshd_map(&tv, a->v, a->B, a->Nk, a->Hkv, dv, a->v_stride))
    return FDMA_ERR_UNSUPPORTED;
  const bool has_bias = a->bias != nullptr;
  if (has_bias) {
    if (!bias_map(&tb, a)) return FDMA_ERR_UNSUPPORTED;
  } else {
    tb = tq;
  }
  FwdParams p{};
  p.B = a->B;
  p.Nq = a->Nq;
  p.Nk = a->Nk;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = a->Hq / a->Hkv;
  p.d = a->d;
  p.dv = dv;
  p.nTq = cdiv(a->Nq, kTile);
  p.nTk = cdiv(a->Nk, kTile);
  p.scale = a->scale;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.test_short_wait = (a->flags & FDMA_FLAG_TEST_SHORT_WAIT) ? 1 : 0;
  p.bias_bsel = a->bias_stride[0] == 0 ? 0 : 1;
  p.bias_hsel = a->bias_stride[1] == 0 ? 0 : 1;
  p.kmap = reinterpret_cast<const int8_t*>(ws + w.kmap);
  p.bits_row = reinterpret_cast<const uint4*>(ws + w.bits_row);
  p.out = static_cast<uint16_t*>(out);
  p.lse = lse;
  p.err = err;
  // up to 128 the kernels run on the padded width (64 or 128) with the missing columns read
  // as zeros; 192 / 128 and 256 / 256 run on the wide kernel at their own widths
  const int run_d = a->d <= 128 ? padded_head_dim(a->d) : a->d;
  const int run_dv = a->d <= 128 ? run_d : dv;
  return launch_fwd(run_d, run_dv, has_bias, tq, tk, tv, tb, p, stream) == cudaSuccess ? FDMA_OK
                                                                                               : FDMA_ERR_CUDA;
}

int fdma_bwd(const fdma_args* a, const void* out, const void* dout, const float* lse, void* dq, void* dk, void* dv,
             void* dbias, void* stream_v) {
  int st = validate(a, false);
  if (st != FDMA_OK) return st;
  st = validate(a, true);
  if (st != FDMA_OK) return st;
  if (out == nullptr || dout == nullptr || lse == nullptr || dq == nullptr || dk == nullptr || dv == nullptr)
    return FDMA_ERR_INVALID;
  if (dbias != nullptr && a->bias == nullptr) return FDMA_ERR_INVALID;
  for (const void* p : {out, dout, static_cast<const void*>(dq), static_cast<const void*>(dk),
                        static_cast<const void*>(dv)})
    if (!aligned16(p)) return FDMA_ERR_UNSUPPORTED;
  if (dbias != nullptr && !aligned16(dbias)) return FDMA_ERR_UNSUPPORTED;
  if (a->workspace_bytes < fdma_workspace_size(a, 1)) return FDMA_ERR_WORKSPACE;
  cudaStream_t stream = static_cast<cudaStream_t>(stream_v);
  int* err = device_error_word();
  if (err == nullptr) return FDMA_ERR_CUDA;
  if (!(a->flags & FDMA_FLAG_REUSE_CLASSIFICATION)) {
    st = classify_into_workspace(a, nullptr, stream);
    if (st != FDMA_OK) return st;
  }
  const WorkspaceLayout w = workspace_layout(a->B, a->Nq, a->Nk, a->Hq, a->Hkv, a->d);
  uint8_t* ws = static_cast<uint8_t*>(a->workspace);
  const int nTq = cdiv(a->Nq, kTile), nTk = cdiv(a->Nk, kTile);
  const int nqpad = nTq * kTile;

  const int dv_w = head_dim_v(*a);
  const bool wide = a->d > 128;  // (192, 128) or (256, 256): the output-split kernels
  BwdPreParams pp{};
  pp.B = a->B;
  pp.Nq = a->Nq;
  pp.Hq = a->Hq;
  pp.d = dv_w;  // delta = <dO, O> over the v head dim
  pp.dpad = dq_acc_width(a->d);
  pp.nqpad = nqpad;
  pp.scale = a->scale;
  pp.out = static_cast<const uint16_t*>(out);
  pp.dout = static_cast<const uint16_t*>(dout);
  pp.lse = lse;
  pp.lse2 = reinterpret_cast<float*>(ws + w.lse2);
  pp.delta = reinterpret_cast<float*>(ws + w.delta);
  pp.dq_acc = reinterpret_cast<float*>(ws + w.dq_acc);
  if (launch_bwd_pre(pp, stream) != cudaSuccess) return FDMA_ERR_CUDA;

  CUtensorMap tq, tk, tv, tdo;
  const int64_t dstr[3] = {static_cast<int64_t>(a->Nq) * a->Hq * dv_w, static_cast<int64_t>(a->Hq) * dv_w, dv_w};
  if (!bshd_map(&tq, a->q, a->B, a->Nq, a->Hq, a->d, a->q_stride) ||
      !bshd_map(&tk, a->k, a->B, a->Nk, a->Hkv, a->d, a->k_stride) ||
      !bshd_map(&tv, a->v, a->B, a->Nk, a->Hkv, dv_w, a->v_stride) ||
      !bshd_map(&tdo, dout, a->B, a->Nq, a->Hq, dv_w, dstr))
    return FDMA_ERR_UNSUPPORTED;
  BwdParams p{};
  p.B = a->B;
  p.Nq = a->Nq;
  p.Nk = a->Nk;
  p.Hq = a->Hq;
  p.Hkv = a->Hkv;
  p.G = a->Hq / a->Hkv;
  p.d = a->d;
  p.nTq = nTq;
  p.nTk = nTk;
  p.nqpad = nqpad;
  p.scale = a->scale;
  p.scale_log2 = a->scale * 1.4426950408889634f;
  p.test_short_wait = (a->flags & FDMA_FLAG_TEST_SHORT_WAIT) ? 1 : 0;
  p.kmap = reinterpret_cast<const int8_t*>(ws + w.kmap);
  p.bits_col = reinterpret_cast<const uint4*>(ws + w.bits_col);
  p.bias = static_cast<const uint16_t*>(a->bias);
  p.bs_b = a->bias_stride[0];
  p.bs_h = a->bias_stride[1];
  p.bs_r = a->bias_stride[2];
  p.bias_bsel = a->bias_stride[0] == 0 ? 0 : 1;
  p.bias_hsel = a->bias_stride[1] == 0 ? 0 : 1;
  p.lse2 = pp.lse2;
  p.delta = pp.delta;
  p.dq_acc = pp.dq_acc;
  p.dk = static_cast<uint16_t*>(dk);
  p.dv = static_cast<uint16_t*>(dv);
  p.dbias = static_cast<uint16_t*>(dbias);
  p.err = err;
  CUtensorMap tb = tq;
  if (a->bias != nullptr) {
    if (!bias_map(&tb, a)) return FDMA_ERR_UNSUPPORTED;
  }
  CUtensorMap tdb = tq;
  if (dbias != nullptr) {
    const uint64_t dims[4] = {static_cast<uint64_t>(a->Nk), static_cast<uint64_t>(a->Nq),
                              static_cast<uint64_t>(a->Hkv), static_cast<uint64_t>(a->B)};
    const uint64_t sb[3] = {static_cast<uint64_t>(a->Nk) * 2, static_cast<uint64_t>(a->Nq) * a->Nk * 2,
                            static_cast<uint64_t>(a->Hkv) * a->Nq * a->Nk * 2};
    if (!make_map(&tdb, dbias, dims, sb)) return FDMA_ERR_UNSUPPORTED;
  }
  const cudaError_t le =
      wide ? launch_bwd_wide(a->d, dv_w, a->bias != nullptr, dbias != nullptr, tq, tk, tv, tdo, tb, p, stream)
           : launch_bwd(padded_head_dim(a->d), a->bias != nullptr, dbias != nullptr, tq, tk, tv, tdo, tb, tdb, p, stream);
  if (le != cudaSuccess) return FDMA_ERR_CUDA;
  DqConvertParams cp{};
  cp.B = a->B;
  cp.Nq = a->Nq;
  cp.Hq = a->Hq;
  cp.d = a->d;
  cp.dpad = dq_acc_width(a->d);
  cp.nqpad = nqpad;
  cp.dq_acc = pp.dq_acc;
  cp.dq = static_cast<uint16_t*>(dq);
  return launch_dq_convert(cp, stream) == cudaSuccess ? FDMA_OK : FDMA_ERR_CUDA;
}

int fdma_get_device_error(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FDMA_ERR_CUDA;
  int* word = device_error_word();
  if (word == nullptr) return FDMA_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, word, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FDMA_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(word, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess) return FDMA_ERR_CUDA;
  }
  return v;
}

const char* fdma_status_string(int s) {
  switch (s) {
    case FDMA_OK:
      return "ok";
    case FDMA_ERR_INVALID:
      return "invalid argument";
    case FDMA_ERR_UNSUPPORTED:
      return "unsupported configuration";
    case FDMA_ERR_CUDA:
      return "CUDA error";
    case FDMA_ERR_TIMEOUT:
      return "device wait timed out";
    case FDMA_ERR_WORKSPACE:
      return "workspace missing or too small";
    default:
      return "unknown status";
  }
}

int fdma_topk_mask(const void* bias, const int64_t bias_stride[3], int B, int Hkv, int Nq, int Nk, int keep_window,
                   int mask_kind, void* mask, void* bias_out, void* stream) {
  if (bias == nullptr || bias_stride == nullptr || mask == nullptr) return FDMA_ERR_INVALID;
  if (B <= 0 || Hkv <= 0 || Nq <= 0 || Nk <= 0 || keep_window <= 0) return FDMA_ERR_INVALID;
  if (mask_kind != FDMA_MASK_DENSE && mask_kind != FDMA_MASK_DENSE_U8) return FDMA_ERR_INVALID;
  if (Nk > kTopkMaxKeys || (Nk & 7) != 0) return FDMA_ERR_UNSUPPORTED;
  for (int a = 0; a < 3; ++a) {
    if (bias_stride[a] < 0) return FDMA_ERR_INVALID;
    if ((bias_stride[a] & 7) != 0) return FDMA_ERR_UNSUPPORTED;
    // written in place or to a buffer of the same layout: rows must not alias
    if (bias_out != nullptr && bias_stride[a] == 0) return FDMA_ERR_INVALID;
  }
  if (bias_out != nullptr && bias_stride[2] < Nk) return FDMA_ERR_INVALID;
  if (!aligned16(bias) || !aligned16(mask) || (bias_out != nullptr && !aligned16(bias_out)))
    return FDMA_ERR_UNSUPPORTED;
  TopkParams p{};
  p.B = B;
  p.Hkv = Hkv;
  p.Nq = Nq;
  p.Nk = Nk;
  p.keep = keep_window;
  for (int a = 0; a < 3; ++a) p.bias_stride[a] = bias_stride[a];
  p.bias = static_cast<const uint16_t*>(bias);
  p.bias_out = static_cast<uint16_t*>(bias_out);
  if (mask_kind == FDMA_MASK_DENSE) p.mask_bf16 = static_cast<uint16_t*>(mask);
  else p.mask_u8 = static_cast<uint8_t*>(mask);
  return launch_topk(p, static_cast<cudaStream_t>(stream)) == cudaSuccess ? FDMA_OK : FDMA_ERR_CUDA;
}

}  // extern "C"
