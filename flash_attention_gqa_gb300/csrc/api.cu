// C ABI of the GB300 blocked GQA flash-attention library: argument checks,
// TMA tensor-map construction, kernel launches and the device status word.
// Every check happens on the host before anything is enqueued; nothing here
// allocates device memory or synchronises (except fa_check_status).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include "../../include/fa.h"
#include "kernels.h"

namespace fa {
// Device error word: bounded waits that give up OR their code in here.
__device__ uint32_t g_fa_error = 0;
}  // namespace fa

namespace {

using fa::kRows;

std::atomic<uint64_t> g_wait_limit_ns{0};
std::atomic<int> g_bwd_kv_rows{0};  // 0: chosen per call; 64 / 128: forced where valid
std::atomic<int> g_bwd_q_splits{0};  // 0: chosen per call; 1..4: forced where a split can apply
std::atomic<int> g_fwd_schedule{0};  // 0: chosen per call; 1: CTA per Q tile; 2: persistent

uint64_t wait_limit() {
  uint64_t v = g_wait_limit_ns.load();
  if (v == 0) {
    v = 2000000000ull;
    if (const char* e = std::getenv("FA_WAIT_LIMIT_NS")) {
      const unsigned long long x = std::strtoull(e, nullptr, 10);
      if (x > 0) v = x;
    }
    g_wait_limit_ns.store(v);
  }
  return v;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    cudaDriverEntryPointQueryResult q;
    void* p = nullptr;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// Device address of the error word on the current device (cached per device).
uint32_t* error_word() {
  static uint32_t* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, fa::g_fa_error) != cudaSuccess) return nullptr;
    addr[dev] = static_cast<uint32_t*>(p);
  }
  return addr[dev];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool pow2_le128(int g) { return g >= 1 && g <= 128 && (g & (g - 1)) == 0; }

// q-like tensor [B*K, G, T, H] as a 4-D map with a box of one Q tile x 64 dims.
bool make_q_map(CUtensorMap* m, const void* ptr, int BK, int G, int T, int H) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)G, (cuuint64_t)BK};
  cuuint64_t strides[3] = {(cuuint64_t)H * 2, (cuuint64_t)T * H * 2, (cuuint64_t)G * T * H * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)(kRows / G), (cuuint32_t)G, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// k-like tensor [B*K, S, H] as a 3-D map with a box of `rows` keys x 64 dims.
bool make_kv_map(CUtensorMap* m, const void* ptr, int BK, int S, int H, int rows) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)BK};
  cuuint64_t strides[2] = {(cuuint64_t)H * 2, (cuuint64_t)S * H * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// k-like tensor [B*K, S, H] viewed as 4-D {64 dims, S, H/64 chunks, B*K} with
// a box of `rows` keys x `chunks` x 64 dims: one copy lands `chunks`
// consecutive [rows x 128 B] swizzled chunks, the layout per-chunk boxes give.
bool make_kv_tile_map(CUtensorMap* m, const void* ptr, int BK, int S, int H, int rows, int chunks) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[4] = {64, (cuuint64_t)S, (cuuint64_t)(H / 64), (cuuint64_t)BK};
  cuuint64_t strides[3] = {(cuuint64_t)H * 2, 128, (cuuint64_t)S * H * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)rows, (cuuint32_t)chunks, 1};
  cuuint32_t es[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(ptr), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared shape checks of the forward and backward passes.
int check_shapes(int B, int K, int G, int T, int S, int H, int causal, const void* seg_q,
                 const void* seg_kv) {
  if (B < 0 || K < 0 || G < 0 || T < 0 || S < 0 || H < 0) return FA_ERR_INVALID_ARG;
  if ((seg_q == nullptr) != (seg_kv == nullptr)) return FA_ERR_INVALID_ARG;
  if (seg_q && (!aligned16(seg_q) || !aligned16(seg_kv))) return FA_ERR_INVALID_ARG;
  (void)causal;
  if (H != 64 && H != 128 && H != 256) return FA_ERR_UNSUPPORTED;
  if (!pow2_le128(G)) return FA_ERR_UNSUPPORTED;
  if ((S + fa::kKvRows - 1) / fa::kKvRows > fa::kMaxKvTiles) return FA_ERR_UNSUPPORTED;
  if ((long long)B * K > 65535) return FA_ERR_UNSUPPORTED;
  if ((long long)T * B * K > (1LL << 31) - 1) return FA_ERR_UNSUPPORTED;  // flat grids
  return FA_OK;
}

}  // namespace

namespace {

size_t splitkv_parts(int B, int K, int G, int T, int H, int n_splits, size_t* o_bytes) {
  const size_t rows = (size_t)B * K * G * T;
  const size_t ob = ((size_t)n_splits * rows * H * sizeof(float) + 255) & ~(size_t)255;
  const size_t lb = ((size_t)n_splits * rows * sizeof(float) + 255) & ~(size_t)255;
  if (o_bytes) *o_bytes = ob;
  return ob + lb;
}

// Checks a block-mask argument set and fills `bm` (cls == nullptr: no mask).
int make_block_mask(fa::BlockMask* bm, const uint8_t* cls, const int32_t* idx, const uint32_t* bits,
                    int heads, int K, int G, int T, int S) {
  *bm = fa::BlockMask{};
  if (cls == nullptr && idx == nullptr && bits == nullptr) return FA_OK;
  if (!cls || !idx || !bits) return FA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(idx) & 3u) || (reinterpret_cast<uintptr_t>(bits) & 3u))
    return FA_ERR_INVALID_ARG;
  if (heads != 1 && heads != K * G) return FA_ERR_INVALID_ARG;
  bm->cls = cls;
  bm->idx = idx;
  bm->bits = bits;
  bm->heads = heads;
  bm->nqb = (T + 127) / 128;
  bm->nkb = (S + 127) / 128;
  return FA_OK;
}

// Shared body of the forward entry points.
int fwd_common(const void* q, const void* k, const void* v, const int32_t* seg_q,
               const int32_t* seg_kv, int causal, void* o, float* lse, const fa::BlockMask& bm,
               int n_splits, void* workspace, size_t workspace_bytes, int B, int K, int G, int T,
               int S, int H, void* stream) {
  const int rc = check_shapes(B, K, G, T, S, H, causal, seg_q, seg_kv);
  if (rc != FA_OK) return rc;
  // Pointers are required (and must be aligned) only for tensors with elements.
  const long rows = (long)B * K * G * T;
  const bool has_kv = (long)B * K * S > 0;
  if (rows > 0 && (!q || !o || !lse || !aligned16(q) || !aligned16(o) ||
                   (reinterpret_cast<uintptr_t>(lse) & 3u) != 0))
    return FA_ERR_INVALID_ARG;
  if (has_kv && (!k || !v || !aligned16(k) || !aligned16(v))) return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (rows == 0) return FA_OK;
  if (S == 0) {
    return fa::launch_fill_empty(o, lse, rows, H, st) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
  }
  size_t o_bytes = 0;
  if (n_splits > 1) {
    const size_t need = splitkv_parts(B, K, G, T, H, n_splits, &o_bytes);
    if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0)
      return FA_ERR_INVALID_ARG;
  }
  fa::FwdArgs a{};
  const int BK = B * K;
  const int cc = fa::fwd_copy_chunks(H);
  if (!make_q_map(&a.tm_q, q, BK, G, T, H) || !make_kv_tile_map(&a.tm_k, k, BK, S, H, fa::kKvRows, cc) ||
      !make_kv_tile_map(&a.tm_v, v, BK, S, H, fa::kKvRows, cc) || !make_q_map(&a.tm_o, o, BK, G, T, H))
    return FA_ERR_CUDA;
  a.o = o;
  a.lse = lse;
  a.seg_q = seg_q;
  a.seg_kv = seg_kv;
  a.B = B; a.K = K; a.G = G; a.T = T; a.S = S; a.H = H;
  a.causal = causal ? 1 : 0;
  a.n_qtiles = (T + kRows / G - 1) / (kRows / G);
  a.bm = bm;
  a.n_splits = n_splits;
  if (n_splits > 1) {
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + o_bytes);
  }
  a.err = error_word();
  a.wait_limit_ns = wait_limit();
  if (!a.err) return FA_ERR_CUDA;
  cudaError_t e = fa::launch_fwd(a, st, g_fwd_schedule.load());
  if (e == cudaSuccess && n_splits > 1)
    e = fa::launch_split_combine(a.part_o, a.part_lse, n_splits, o, lse, rows, H, st);
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, const int32_t* seg_q,
           const int32_t* seg_kv, int causal, void* o, float* lse, int B, int K, int G, int T,
           int S, int H, void* stream) {
  return fwd_common(q, k, v, seg_q, seg_kv, causal, o, lse, fa::BlockMask{}, 1, nullptr, 0, B, K,
                    G, T, S, H, stream);
}

int fa_fwd_masked(const void* q, const void* k, const void* v, const int32_t* seg_q,
                  const int32_t* seg_kv, int causal, const uint8_t* block_class,
                  const int32_t* partial_index, const uint32_t* partial_bits, int mask_heads,
                  void* o, float* lse, int B, int K, int G, int T, int S, int H, void* stream) {
  fa::BlockMask bm;
  const int rc = make_block_mask(&bm, block_class, partial_index, partial_bits, mask_heads, K, G, T, S);
  if (rc != FA_OK) return rc;
  return fwd_common(q, k, v, seg_q, seg_kv, causal, o, lse, bm, 1, nullptr, 0, B, K, G, T, S, H,
                    stream);
}

size_t fa_fwd_splitkv_workspace_size(int B, int K, int G, int T, int S, int H, int n_splits) {
  if (B <= 0 || K <= 0 || G <= 0 || T <= 0 || S < 0 || n_splits < 1 || n_splits > 256) return 0;
  if (check_shapes(B, K, G, T, S, H, 0, nullptr, nullptr) != FA_OK) return 0;
  return splitkv_parts(B, K, G, T, H, n_splits, nullptr);
}

int fa_fwd_splitkv_default_splits(int B, int K, int G, int T, int S, int H) {
  if (B <= 0 || K <= 0 || G <= 0 || T <= 0 || S <= 0) return 1;
  if (check_shapes(B, K, G, T, S, H, 0, nullptr, nullptr) != FA_OK) return 1;
  const long ctas = (long)((T + kRows / G - 1) / (kRows / G)) * B * K;
  const int sms = fa_device_sm_count();
  const int kv_tiles = (S + fa::kKvRows - 1) / fa::kKvRows;
  // Splitting costs partial writes and a merge: only worth it when the Q
  // tiles alone leave SMs idle.  Then as many splits as fit in one wave: a
  // sweep of 1-64 splits on decode shapes (8-64 kv heads, S = 8K-32K, H = 128
  // and 256) put the fastest count at or within 5% of floor(SMs / CTAs); a
  // second, partial wave costs more than it adds.
  long n = (sms > 0 && ctas < sms) ? sms / ctas : 1;
  n = n < 1 ? 1 : n;
  n = n > kv_tiles ? kv_tiles : n;
  return (int)(n > 64 ? 64 : n);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, const int32_t* seg_q,
                   const int32_t* seg_kv, int causal, void* o, float* lse, int n_splits,
                   void* workspace, size_t workspace_bytes, int B, int K, int G, int T, int S, int H,
                   void* stream) {
  if (n_splits < 1 || n_splits > 256) return FA_ERR_INVALID_ARG;
  return fwd_common(q, k, v, seg_q, seg_kv, causal, o, lse, fa::BlockMask{}, n_splits, workspace,
                    workspace_bytes, B, K, G, T, S, H, stream);
}

size_t fa_bwd_workspace_size(int B, int K, int G, int T, int S, int H) {
  if (B <= 0 || K <= 0 || G <= 0 || T <= 0 || S < 0) return 0;
  if (check_shapes(B, K, G, T, S, H, 0, nullptr, nullptr) != FA_OK) return 0;
  return fa::bwd_workspace(B, K, G, T, S, H, fa_device_sm_count()).total;
}

namespace {

// Shared body of fa_bwd and fa_bwd_stage: stage < 0 runs every stage.  The
// workspace must hold the base part; the Q-range split of a dK/dV grid smaller
// than the GPU runs where allow_split and the workspace also holds the split part.
int bwd_impl(int stage, const void* q, const void* k, const void* v, const void* o, const float* lse,
             const void* dO, const int32_t* seg_q, const int32_t* seg_kv, int causal,
             const fa::BlockMask& bm, void* dq, void* dk, void* dv, void* workspace,
             size_t workspace_bytes, int B, int K, int G, int T, int S, int H, void* stream,
             bool allow_split) {
  if (stage < -1 || stage > 2) return FA_ERR_INVALID_ARG;
  const int rc = check_shapes(B, K, G, T, S, H, causal, seg_q, seg_kv);
  if (rc != FA_OK) return rc;
  // Pointers are required (and must be aligned) only for tensors with elements.
  const bool has_rows = (long)B * K * G * T > 0;
  const bool has_kv = (long)B * K * S > 0;
  if (has_rows && (!q || !o || !lse || !dO || !dq || !aligned16(q) || !aligned16(o) ||
                   !aligned16(dO) || !aligned16(dq) || !aligned16(lse)))
    return FA_ERR_INVALID_ARG;
  if (has_kv && (!k || !v || !dk || !dv || !aligned16(k) || !aligned16(v) || !aligned16(dk) ||
                 !aligned16(dv)))
    return FA_ERR_INVALID_ARG;
  const int sms = fa_device_sm_count();
  const fa::BwdWorkspace wl = fa::bwd_workspace(B, K, G, T, S, H, sms);
  if ((long)B * K * G * T > 0 && (workspace == nullptr || workspace_bytes < wl.base ||
                                  (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0))
    return FA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const long rows = (long)B * K * G * T;
  const int BK = B * K;
  const int forced = g_bwd_kv_rows.load();
  const int kvr = (H <= 128 && forced != 0) ? forced : fa::bwd_kv_rows(H, B, K, S, sms);
  if (BK == 0) return FA_OK;
  if (rows == 0 || S == 0) {
    // No query rows or no keys: every gradient is zero.
    if ((stage < 0 || stage == 2) && rows > 0 &&
        cudaMemsetAsync(dq, 0, (size_t)rows * H * 2, st) != cudaSuccess)
      return FA_ERR_CUDA;
    if ((stage < 0 || stage == 1) && S > 0 &&
        (cudaMemsetAsync(dk, 0, (size_t)BK * S * H * 2, st) != cudaSuccess ||
         cudaMemsetAsync(dv, 0, (size_t)BK * S * H * 2, st) != cudaSuccess))
      return FA_ERR_CUDA;
    return FA_OK;
  }
  fa::BwdArgs a{};
  if (!make_q_map(&a.tm_q, q, BK, G, T, H) || !make_q_map(&a.tm_do, dO, BK, G, T, H) ||
      !make_kv_map(&a.tm_k, k, BK, S, H, kvr) || !make_kv_map(&a.tm_v, v, BK, S, H, kvr) ||
      !make_q_map(&a.tm_dq, dq, BK, G, T, H))
    return FA_ERR_CUDA;
  float* delta = static_cast<float*>(workspace);
  // The range table starts at its own 256-byte boundary past the D rows (an
  // offset of rows * 4 bytes would misalign its 8-byte pairs for odd row counts).
  int2* ranges = reinterpret_cast<int2*>(static_cast<char*>(workspace) + wl.ranges);
  if ((reinterpret_cast<uintptr_t>(ranges) & 7u) != 0) return FA_ERR_INVALID_ARG;
  a.lse = lse;
  a.delta = delta;
  a.seg_ranges = ranges;
  a.seg_runs = reinterpret_cast<uint8_t*>(static_cast<char*>(workspace) + wl.runs);
  a.dq = dq; a.dk = dk; a.dv = dv;
  a.seg_q = seg_q; a.seg_kv = seg_kv;
  a.B = B; a.K = K; a.G = G; a.T = T; a.S = S; a.H = H;
  a.causal = causal ? 1 : 0;
  a.n_qtiles = (T + kRows / G - 1) / (kRows / G);
  a.n_kvtiles = (S + kvr - 1) / kvr;
  a.kv_rows = kvr;
  const long dkdv_ctas = (long)BK * a.n_kvtiles;
  // Split counters exist wherever the workspace holds the split part; stage 0
  // zeroes them then (the last CTA of each KV tile re-zeroes its own after use).
  const bool split_ok = allow_split && wl.partials > 0 && workspace_bytes >= wl.total && dkdv_ctas < sms;
  int* counters = split_ok ? reinterpret_cast<int*>(static_cast<char*>(workspace) + wl.counters) : nullptr;
  a.q_splits = 1;
  if (split_ok) {
    const int fs = g_bwd_q_splits.load();
    const bool uneven = causal || seg_q != nullptr || bm.cls != nullptr;
    a.q_splits = fs != 0 ? fs : fa::bwd_q_splits(dkdv_ctas, sms, uneven, H);
  }
  if (a.q_splits > 1) {
    a.dkv_count = counters;
    a.dkv_part = reinterpret_cast<float*>(static_cast<char*>(workspace) + wl.partials);
  }
  a.bm = bm;
  a.err = error_word();
  a.wait_limit_ns = wait_limit();
  if (!a.err) return FA_ERR_CUDA;
  cudaError_t e = cudaSuccess;
  if (stage < 0 || stage == 0) {
    e = fa::launch_bwd_preprocess(o, dO, delta, rows, H, counters, (int)dkdv_ctas, st);
    if (e == cudaSuccess) e = fa::launch_seg_ranges(a, st);
  }
  if (e == cudaSuccess && (stage < 0 || stage == 1)) e = fa::launch_bwd_dkdv(a, st);
  // All stages in one call: the dQ grid directly follows the dK/dV grid and may
  // overlap its tail (both read only stage 0's results and the inputs).
  if (e == cudaSuccess && (stage < 0 || stage == 2)) e = fa::launch_bwd_dq(a, st, stage < 0);
  if (e == cudaErrorNotSupported) return FA_ERR_UNSUPPORTED;
  return e == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}

}  // namespace

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const float* lse,
           const void* dO, const int32_t* seg_q, const int32_t* seg_kv, int causal, void* dq,
           void* dk, void* dv, void* workspace, size_t workspace_bytes, int B, int K, int G, int T,
           int S, int H, void* stream) {
  return bwd_impl(-1, q, k, v, o, lse, dO, seg_q, seg_kv, causal, fa::BlockMask{}, dq, dk, dv,
                  workspace, workspace_bytes, B, K, G, T, S, H, stream, true);
}

int fa_bwd_masked(const void* q, const void* k, const void* v, const void* o, const float* lse,
                  const void* dO, const int32_t* seg_q, const int32_t* seg_kv, int causal,
                  const uint8_t* block_class, const int32_t* partial_index,
                  const uint32_t* partial_bits, int mask_heads, void* dq, void* dk, void* dv,
                  void* workspace, size_t workspace_bytes, int B, int K, int G, int T, int S, int H,
                  void* stream) {
  fa::BlockMask bm;
  const int rc = make_block_mask(&bm, block_class, partial_index, partial_bits, mask_heads, K, G, T, S);
  if (rc != FA_OK) return rc;
  return bwd_impl(-1, q, k, v, o, lse, dO, seg_q, seg_kv, causal, bm, dq, dk, dv, workspace,
                  workspace_bytes, B, K, G, T, S, H, stream, true);
}

int fa_block_mask_build(const uint8_t* dense, int heads, int T, int S, uint8_t* block_class,
                        int32_t* partial_index, uint32_t* partial_bits, int64_t partial_capacity,
                        int64_t* n_partial) {
  if (!dense || !block_class || !partial_index || !n_partial || heads < 1 || T < 1 || S < 1 ||
      partial_capacity < 0 || (partial_capacity > 0 && !partial_bits))
    return FA_ERR_INVALID_ARG;
  const int nqb = (T + 127) / 128, nkb = (S + 127) / 128;
  int64_t count = 0;
  for (int h = 0; h < heads; ++h) {
    for (int qb = 0; qb < nqb; ++qb) {
      for (int kb = 0; kb < nkb; ++kb) {
        const int t0 = qb * 128, t1 = t0 + 128 < T ? t0 + 128 : T;
        const int s0 = kb * 128, s1 = s0 + 128 < S ? s0 + 128 : S;
        long kept = 0;
        for (int t = t0; t < t1; ++t) {
          const uint8_t* row = dense + ((long)h * T + t) * S;
          for (int s = s0; s < s1; ++s) kept += row[s] != 0;
        }
        const long total = (long)(t1 - t0) * (s1 - s0);
        const long blk = ((long)h * nqb + qb) * nkb + kb;
        partial_index[blk] = -1;
        if (kept == 0) {
          block_class[blk] = 0;  // EMPTY: the kernels skip the tile
        } else if (kept == total) {
          block_class[blk] = 1;  // FULL: no per-element mask
        } else {
          block_class[blk] = 2;  // PARTIAL: 128 x 128 bits, row-major, 4 words per row
          if (count < partial_capacity) {
            uint32_t* bits = partial_bits + count * 128 * 4;
            for (int i = 0; i < 128 * 4; ++i) bits[i] = 0;
            for (int t = t0; t < t1; ++t) {
              const uint8_t* row = dense + ((long)h * T + t) * S;
              for (int s = s0; s < s1; ++s)
                if (row[s]) bits[(t - t0) * 4 + (s - s0) / 32] |= 1u << ((s - s0) % 32);
            }
          }
          partial_index[blk] = (int32_t)count;
          ++count;
        }
      }
    }
  }
  *n_partial = count;
  if (partial_bits != nullptr && count > partial_capacity) return FA_ERR_INVALID_ARG;
  return FA_OK;
}

int fa_bwd_stage(int stage, const void* q, const void* k, const void* v, const void* o,
                 const float* lse, const void* dO, const int32_t* seg_q, const int32_t* seg_kv,
                 int causal, void* dq, void* dk, void* dv, void* workspace, size_t workspace_bytes,
                 int B, int K, int G, int T, int S, int H, void* stream) {
  if (stage < 0) return FA_ERR_INVALID_ARG;
  return bwd_impl(stage, q, k, v, o, lse, dO, seg_q, seg_kv, causal, fa::BlockMask{}, dq, dk, dv,
                  workspace, workspace_bytes, B, K, G, T, S, H, stream, true);
}

// ------------------------------------------------------------------------
// fa_bwd_noalloc: fa_bwd for callers that may not allocate device memory.
// Its scratch is this fixed array; the host only ever uses the array's device
// address, looked up once per device with that device current.
static __device__ __align__(256) unsigned char g_bwd_noalloc_scratch[FA_NOALLOC_SCRATCH_BYTES];

namespace {

void* noalloc_scratch_address() {
  static void* addr[64] = {};
  static std::mutex mu;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
  std::lock_guard<std::mutex> lk(mu);
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_bwd_noalloc_scratch) != cudaSuccess || p == nullptr)
      return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

int fa_bwd_noalloc(const void* q, const void* k, const void* v, const void* o, const float* lse,
                   const void* dO, const int32_t* seg_q, const int32_t* seg_kv, int causal,
                   void* dq, void* dk, void* dv, int B, int K, int G, int T, int S, int H,
                   void* stream) {
  const int rc = check_shapes(B, K, G, T, S, H, causal, seg_q, seg_kv);
  if (rc != FA_OK) return rc;
  // Only the base part (D rows, segment tables) lives in the scratch: no Q-range split here.
  if (fa::bwd_workspace(B, K, G, T, S, H, 0).base > (size_t)FA_NOALLOC_SCRATCH_BYTES)
    return FA_ERR_UNSUPPORTED;
  void* scratch = noalloc_scratch_address();
  if (scratch == nullptr) return FA_ERR_CUDA;
  return bwd_impl(-1, q, k, v, o, lse, dO, seg_q, seg_kv, causal, fa::BlockMask{}, dq, dk, dv,
                  scratch, (size_t)FA_NOALLOC_SCRATCH_BYTES, B, K, G, T, S, H, stream, false);
}

int fa_check_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return FA_ERR_CUDA;
  uint32_t err = 0;
  if (cudaMemcpyFromSymbol(&err, fa::g_fa_error, sizeof(err)) != cudaSuccess) return FA_ERR_CUDA;
  if (err != 0) {
    const uint32_t zero = 0;
    if (cudaMemcpyToSymbol(fa::g_fa_error, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_CUDA;
    return FA_ERR_DEVICE_TIMEOUT;
  }
  return FA_OK;
}

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported shape or option";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_DEVICE_TIMEOUT: return "a bounded device wait timed out";
    default: return "unknown status";
  }
}

int fa_set_wait_limit_ns(uint64_t ns) {
  if (ns == 0) return FA_ERR_INVALID_ARG;
  g_wait_limit_ns.store(ns);
  return FA_OK;
}

int fa_set_bwd_kv_rows(int rows) {
  if (rows != 0 && rows != 64 && rows != 128) return FA_ERR_INVALID_ARG;
  g_bwd_kv_rows.store(rows);
  return FA_OK;
}

int fa_set_bwd_q_splits(int n) {
  if (n < 0 || n > fa::kMaxQSplits) return FA_ERR_INVALID_ARG;
  g_bwd_q_splits.store(n);
  return FA_OK;
}

int fa_bwd_plan(int B, int K, int G, int T, int S, int H, int causal, int masked, int sm_count,
                int* kv_rows, int* q_splits) {
  if (kv_rows == nullptr || q_splits == nullptr || sm_count < 0) return FA_ERR_INVALID_ARG;
  const int rc = check_shapes(B, K, G, T, S, H, causal, nullptr, nullptr);
  if (rc != FA_OK) return rc;
  const int kvr = fa::bwd_kv_rows(H, B, K, S, sm_count);
  const long ctas = (long)B * K * ((S + kvr - 1) / kvr);
  *kv_rows = kvr;
  *q_splits = fa::bwd_q_splits(ctas, sm_count, causal != 0 || masked != 0, H);
  return FA_OK;
}

int fa_set_fwd_schedule(int mode) {
  if (mode < 0 || mode > 2) return FA_ERR_INVALID_ARG;
  g_fwd_schedule.store(mode);
  return FA_OK;
}

int fa_selftest_wait_timeout(void* stream) {
  uint32_t* err = error_word();
  if (!err) return FA_ERR_CUDA;
  if (fa::launch_wait_selftest(err, wait_limit(), static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_CUDA;
  return fa_check_status(stream);
}

int fa_device_sm_count(void) {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return n;
}

}  // extern "C"
