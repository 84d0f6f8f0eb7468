// Host side of the C ABI declared in include/fa.h: argument validation,
// tensor-map encoding, kernel selection and launch, for the forward pass
// (single pass and split-KV) and the backward pass.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "fa.h"
#include "fa_bwd_kernel.cuh"
#include "fa_fp8.cuh"
#include "fa_fwd_kernel.cuh"
#include "fa_merge.cuh"

namespace fa {

__device__ unsigned int g_status;  // wait-site bits; nonzero = a wait gave up

namespace {

constexpr int kMaxDevices = 64;
unsigned long long g_timeout_ns = 1000000000ull;
int g_test_withhold_q = 0;

// cuTensorMapEncodeTiled, fetched from the driver through the runtime so the
// library does not link libcuda directly.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

// [BH, L, D] bf16 viewed as a 3-D tensor (innermost first: D, L, BH) with a
// 64 x 128 x 1 box and the 128-byte swizzle.  Rows past L inside a head are
// out of bounds and read as zeros; they never spill into the next head.
bool encode_map(CUtensorMap* map, const void* ptr, int BH, int L, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2,
                                 static_cast<cuuint64_t>(L) * D * 2};
  const cuuint32_t box[3] = {64, static_cast<cuuint32_t>(BLOCK_N), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// E4M3 codes [BH, L, D] (one byte each) as a 3-D tensor (D, L, BH) with a
// D x 128 x 1 box: one box per 128-row tile, rows of D bytes, 128-byte
// swizzle at D = 128 and 64-byte swizzle at D = 64 (the layouts the FP8
// MMA descriptors read).
bool encode_map_u8(CUtensorMap* map, const void* ptr, int BH, int L, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L) * D};
  const cuuint32_t box[3] = {static_cast<cuuint32_t>(D), static_cast<cuuint32_t>(BLOCK_N), 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void*>(ptr), dims, strides, box,
            estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            D == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The fp32 dQ accumulator [BH, L, D] as a 3-D tensor (D, L, BH) with a
// 32 x 128 x 1 box (128-byte rows, one query block's rows of a 32-column
// strip) and the 128-byte swizzle: the target of the backward kernel's
// reduce-adds.  Rows past L inside a head are out of bounds, so a reduce of
// a ragged block never touches the next head.
bool encode_map_f32_acc(CUtensorMap* map, void* ptr, int BH, int L, int D) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(L),
                              static_cast<cuuint64_t>(BH)};
  const cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 4,
                                 static_cast<cuuint64_t>(L) * D * 4};
  const cuuint32_t box[3] = {32, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, ptr, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <typename Kernel>
bool configure_once(Kernel kernel, int smem, int dev, bool* configured, std::mutex& mu) {
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= kMaxDevices) return false;
  if (!configured[dev]) {
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return false;
    configured[dev] = true;
  }
  return true;
}

// Multiprocessor count of device `dev`, queried once (0 if the query fails).
int sm_count(int dev) {
  static int count[kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= kMaxDevices) return 0;
  if (count[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    count[dev] = n;
  }
  return count[dev];
}

template <int D, bool CAUSAL, bool SPLIT, bool FP8 = false>
int launch(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
           const FwdArgs& args, int n_splits, cudaStream_t stream, int dev) {
  auto kernel = fa_fwd_kernel<D, CAUSAL, SPLIT, FP8>;
  constexpr int smem = FwdCfg<D, FP8>::SMEM_BYTES;
  static bool configured[kMaxDevices] = {};
  static std::mutex mu;
  if (!configure_once(kernel, smem, dev, configured, mu)) return FA_ERR_LAUNCH;
  const dim3 grid(static_cast<unsigned>(args.n_ctiles) * static_cast<unsigned>(args.bh) *
                  static_cast<unsigned>(n_splits));
  kernel<<<grid, FwdCfg<D, FP8>::THREADS, smem, stream>>>(mq, mk, mv, args);
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

// Launch `kernel` as a programmatic dependant of the previous work on
// `stream` (it may start while that work drains and must wait for it with
// griddepcontrol.wait before reading its results).
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                             cudaStream_t stream, Args... args) {
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

template <int D>
int launch_merge(const FwdArgs& args, int n_splits, cudaStream_t stream) {
  const int64_t rows = static_cast<int64_t>(args.bh) * args.L;
  const dim3 grid(static_cast<unsigned>((rows + MERGE_WARPS - 1) / MERGE_WARPS));
  // a programmatic dependant of the split pass: launched while it drains,
  // it waits for that grid before reading the partials
  const float* o_part = args.o_part;
  const float* lse_part = args.lse_part;
  return launch_dependent(fa_merge_kernel<D>, grid, dim3(MERGE_WARPS * 32), 0, stream, o_part,
                          lse_part, args.o, args.lse, rows, n_splits) == cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Validation shared by every entry point, then the tensor maps and kernel
// arguments.  Returns FA_OK or the status of the first failed check; nothing
// is launched here.
struct Prepared {
  CUtensorMap mq, mk, mv;
  FwdArgs args;
  int dev;
};

int prepare(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int L,
            int d, float scale, int causal, Prepared* out) {
  if (!q || !k || !v || !o || !lse) return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || L < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t n_ct = (static_cast<int64_t>(L) + ROWS_PER_CTA - 1) / ROWS_PER_CTA;
  if (BH > 0x7fffffff || BH * n_ct > 0x7fffffff) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(lse, 4))
    return FA_ERR_MISALIGNED;

  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_DEVICE;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;

  if (!encode_map(&out->mq, q, static_cast<int>(BH), L, d) ||
      !encode_map(&out->mk, k, static_cast<int>(BH), L, d) ||
      !encode_map(&out->mv, v, static_cast<int>(BH), L, d))
    return FA_ERR_LAUNCH;

  unsigned int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status) != cudaSuccess)
    return FA_ERR_LAUNCH;

  FwdArgs& args = out->args;
  args.o = static_cast<uint16_t*>(o);
  args.lse = lse;
  args.blocks_per_split = 0;
  args.o_part = nullptr;
  args.lse_part = nullptr;
  args.L = L;
  args.n_ctiles = static_cast<int>(n_ct);
  args.bh = static_cast<int>(BH);
  {
    // Heads per scheduling group: K + V of a group within ~32 MB of L2.
    const int64_t kv_bytes = static_cast<int64_t>(L) * d * 2 * 2;
    const int64_t g = kv_bytes > 0 ? (int64_t{32} << 20) / kv_bytes : BH;
    args.group_heads = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  }
  args.scale_log2 = scale * 1.4426950408889634f;
  args.q_scale = nullptr;
  args.k_scale = nullptr;
  args.n_blocks = static_cast<int>((static_cast<int64_t>(L) + BLOCK_N - 1) / BLOCK_N);
  args.status = status;
  args.timeout_ns = g_timeout_ns;
  args.test_withhold_q = g_test_withhold_q;
  out->dev = dev;
  return FA_OK;
}

// Effective split count: no more splits than K/V blocks, and no split left
// without a block (blocks_per_split = ceil(blocks / splits)).
void split_plan(int L, int n_splits, int* eff_splits, int* blocks_per_split) {
  const int blocks = (L + BLOCK_N - 1) / BLOCK_N;
  int ns = n_splits < blocks ? n_splits : blocks;
  const int bps = (blocks + ns - 1) / ns;
  ns = (blocks + bps - 1) / bps;
  *eff_splits = ns;
  *blocks_per_split = bps;
}

constexpr int kMaxSplits = 64;

size_t align256(size_t x) { return (x + 255) & ~size_t{255}; }

// Workspace of the split pass for the split count actually used
// (split_plan's effective count, never more than the requested one).
size_t workspace_bytes(int64_t BH, int L, int d, int n_splits) {
  int ns = 1, bps = 1;
  split_plan(L, n_splits, &ns, &bps);
  const size_t rows = static_cast<size_t>(BH) * static_cast<size_t>(L);
  return align256(static_cast<size_t>(ns) * rows * d * 4) + static_cast<size_t>(ns) * rows * 4;
}

// ---------------------------------------------------------------- backward
// Workspace of the backward pass: fp32 dQ accumulator [BH, L, d], then the
// per-query terms -lse*log2(e) and -scale*<dO_i, O_i>, each [BH, Lp] with
// Lp = L rounded up to 128, every part 256-byte aligned.
struct BwdLayout {
  size_t acc_bytes, row_bytes, total;  // the unit counter sits in the last 256 bytes
};

BwdLayout bwd_layout(int64_t BH, int L, int d) {
  const size_t Lp = (static_cast<size_t>(L) + 127) / 128 * 128;
  BwdLayout w;
  w.acc_bytes = align256(static_cast<size_t>(BH) * static_cast<size_t>(L) * d * 4);
  w.row_bytes = align256(static_cast<size_t>(BH) * Lp * 4);
  w.total = w.acc_bytes + 2 * w.row_bytes + 256;
  return w;
}

template <int D, bool CAUSAL>
int launch_bwd(const CUtensorMap& mq, const CUtensorMap& mk, const CUtensorMap& mv,
               const CUtensorMap& mdo, const CUtensorMap& mdq, const BwdArgs& args,
               const BwdPreArgs& pre, uint16_t* dq, cudaStream_t stream, int dev) {
  auto kernel = fa_bwd_kernel<D, CAUSAL>;
  constexpr int smem = BwdCfg<D>::SMEM_BYTES;
  static bool configured[kMaxDevices] = {};
  static std::mutex mu;
  if (!configure_once(kernel, smem, dev, configured, mu)) return FA_ERR_LAUNCH;
  constexpr long long pre_rows_per_block = BWD_AUX_WARPS * BWD_PRE_ROWS;
  const dim3 pre_grid(
      static_cast<unsigned>((pre.rows + pre_rows_per_block - 1) / pre_rows_per_block));
  fa_bwd_pre_kernel<D><<<pre_grid, BWD_AUX_WARPS * 32, 0, stream>>>(pre);
  if (cudaGetLastError() != cudaSuccess) return FA_ERR_LAUNCH;
  // The gradient kernel and the post-pass are programmatic dependants of the
  // kernel before them: each starts while that one drains and waits for it
  // before reading its results.  The gradient kernel is persistent: one CTA
  // per SM (its shared memory admits no second), each taking units until
  // none is left.
  const int sms = sm_count(dev);
  if (sms <= 0) return FA_ERR_DEVICE;
  const dim3 grid(static_cast<unsigned>(args.n_units < sms ? args.n_units : sms));
  if (launch_dependent(kernel, grid, dim3(BwdCfg<D>::THREADS), smem, stream, mq, mk, mv, mdo, mdq,
                       args) != cudaSuccess)
    return FA_ERR_LAUNCH;
  const long long n4 = static_cast<long long>(args.bh) * args.L * D / 4;
  const long long blocks = (n4 + 255) / 256;
  const dim3 post_grid(static_cast<unsigned>(blocks < 152 * 4 ? blocks : 152 * 4));
  const float* acc = args.dq_acc;
  return launch_dependent(fa_bwd_post_kernel, post_grid, dim3(256), 0, stream, acc, dq, n4) ==
                 cudaSuccess
             ? FA_OK
             : FA_ERR_LAUNCH;
}

}  // namespace
}  // namespace fa

// ------------------------------------------------------------------------
// Split-KV without caller-provided scratch.
//
// Some callers cannot allocate device memory at the point where they run
// attention: a serving engine or plugin host that owns the whole device
// memory budget and hands out no workspace, or code whose allocator must not
// be bypassed.  For them the library carries its own split-KV scratch: a
// fixed FA_STATIC_WORKSPACE_BYTES array in device global memory, created
// with the module on every GPU that loads this library and kept until the
// process exits.  The entry point below calls no allocation routine.  On the
// first call on a device it looks up that device's address of the array
// (cudaGetSymbolAddress, with the device current) and remembers it; make
// that first call before any stream capture.  All calls share the one array
// and it keeps whatever the previous call left there: nothing in it has to
// start at zero (the split pass writes every partial the merge reads), but
// calls that overlap on the GPU -- on different streams, or from different
// host threads -- race on it.
static __device__ __align__(256) unsigned char g_splitkv_static_ws[FA_STATIC_WORKSPACE_BYTES];

namespace {

void* static_workspace_address(int dev) {
  static void* addr[fa::kMaxDevices] = {};
  static std::mutex mu;
  std::lock_guard<std::mutex> lock(mu);
  if (dev < 0 || dev >= fa::kMaxDevices) return nullptr;
  if (!addr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_splitkv_static_ws) != cudaSuccess) return nullptr;
    addr[dev] = p;
  }
  return addr[dev];
}

}  // namespace

extern "C" {

int fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H, int L,
           int d, float scale, int causal, fa_stream_t stream) {
  using namespace fa;
  Prepared p;
  const int rc = prepare(q, k, v, o, lse, B, H, L, d, scale, causal, &p);
  if (rc != FA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d == 64)
    return causal ? launch<64, true, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                  : launch<64, false, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
  return causal ? launch<128, true, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                : launch<128, false, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
}

int fa_splitkv_splits(int B, int H, int L, int d, int causal, int num_sms) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128) || (causal != 0 && causal != 1))
    return 0;
  if (num_sms <= 0) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        num_sms <= 0)
      return 0;
  }
  const int64_t ctas = static_cast<int64_t>(B) * H *
                       ((static_cast<int64_t>(L) + fa::ROWS_PER_CTA - 1) / fa::ROWS_PER_CTA);
  const int64_t blocks = (static_cast<int64_t>(L) + fa::BLOCK_N - 1) / fa::BLOCK_N;
  int64_t s = static_cast<int64_t>(num_sms) * (causal ? 2 : 1) / ctas;
  const int64_t cap = blocks < fa::kMaxSplits ? blocks : fa::kMaxSplits;
  s = s < 1 ? 1 : (s > cap ? cap : s);
  return static_cast<int>(s);
}

size_t fa_splitkv_workspace_bytes(int B, int H, int L, int d, int n_splits) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128) || n_splits < 1 ||
      n_splits > fa::kMaxSplits)
    return 0;
  return fa::workspace_bytes(static_cast<int64_t>(B) * H, L, d, n_splits);
}

int fa_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                   int L, int d, float scale, int causal, int n_splits, void* workspace,
                   size_t workspace_bytes_given, fa_stream_t stream) {
  using namespace fa;
  if (n_splits < 1 || n_splits > kMaxSplits || !workspace) return FA_ERR_INVALID_ARG;
  if (B >= 1 && H >= 1 && L >= 1 && (d == 64 || d == 128)) {
    if (workspace_bytes_given < workspace_bytes(static_cast<int64_t>(B) * H, L, d, n_splits))
      return FA_ERR_INVALID_ARG;
    if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  }
  Prepared p;
  const int rc = prepare(q, k, v, o, lse, B, H, L, d, scale, causal, &p);
  if (rc != FA_OK) return rc;
  int ns = 1, bps = 1;
  split_plan(L, n_splits, &ns, &bps);
  if (static_cast<int64_t>(p.args.bh) * p.args.n_ctiles * ns > 0x7fffffff)
    return FA_ERR_INVALID_ARG;
  const size_t rows = static_cast<size_t>(p.args.bh) * static_cast<size_t>(L);
  p.args.blocks_per_split = bps;
  p.args.o_part = static_cast<float*>(workspace);
  p.args.lse_part = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                             align256(static_cast<size_t>(ns) * rows * d * 4));
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  int r;
  if (d == 64)
    r = causal ? launch<64, true, true>(p.mq, p.mk, p.mv, p.args, ns, s, p.dev)
               : launch<64, false, true>(p.mq, p.mk, p.mv, p.args, ns, s, p.dev);
  else
    r = causal ? launch<128, true, true>(p.mq, p.mk, p.mv, p.args, ns, s, p.dev)
               : launch<128, false, true>(p.mq, p.mk, p.mv, p.args, ns, s, p.dev);
  if (r != FA_OK) return r;
  return d == 64 ? launch_merge<64>(p.args, ns, s) : launch_merge<128>(p.args, ns, s);
}

int fa_fwd_splitkv_static(const void* q, const void* k, const void* v, void* o, float* lse,
                          int B, int H, int L, int d, float scale, int causal, int n_splits,
                          fa_stream_t stream) {
  using namespace fa;
  if (n_splits < 1 || n_splits > kMaxSplits) return FA_ERR_INVALID_ARG;
  // The scratch the call will use (for the effective split count) must fit.
  if (B >= 1 && H >= 1 && L >= 1 && (d == 64 || d == 128) &&
      workspace_bytes(static_cast<int64_t>(B) * H, L, d, n_splits) > FA_STATIC_WORKSPACE_BYTES)
    return FA_ERR_INVALID_ARG;  // the sizes need more scratch than the static array holds
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_DEVICE;
  void* ws = static_workspace_address(dev);
  if (!ws) return FA_ERR_LAUNCH;
  return fa_fwd_splitkv(q, k, v, o, lse, B, H, L, d, scale, causal, n_splits, ws,
                        FA_STATIC_WORKSPACE_BYTES, stream);
}

size_t fa_bwd_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128)) return 0;
  return fa::bwd_layout(static_cast<int64_t>(B) * H, L, d).total;
}

int fa_bwd(const void* q, const void* k, const void* v, const void* o, const void* dout,
           const float* lse, void* dq, void* dk, void* dv, int B, int H, int L, int d, float scale,
           int causal, void* workspace, size_t workspace_bytes_given, fa_stream_t stream) {
  using namespace fa;
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !workspace)
    return FA_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || L < 1) return FA_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return FA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t n_kv = (static_cast<int64_t>(L) + 127) / 128;
  if (BH > 0x7fffffff || BH * n_kv > 0x7fffffff ||
      (BH * n_kv * 128 + BWD_AUX_WARPS - 1) / BWD_AUX_WARPS > 0x7fffffff)
    return FA_ERR_INVALID_ARG;
  const BwdLayout w = bwd_layout(BH, L, d);
  if (workspace_bytes_given < w.total) return FA_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(dout, 16) || !aligned(dq, 16) || !aligned(dk, 16) || !aligned(dv, 16) ||
      !aligned(lse, 4) || !aligned(workspace, 256))
    return FA_ERR_MISALIGNED;

  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_DEVICE;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;

  CUtensorMap mq, mk, mv, mdo;
  if (!encode_map(&mq, q, static_cast<int>(BH), L, d) ||
      !encode_map(&mk, k, static_cast<int>(BH), L, d) ||
      !encode_map(&mv, v, static_cast<int>(BH), L, d) ||
      !encode_map(&mdo, dout, static_cast<int>(BH), L, d))
    return FA_ERR_LAUNCH;
  unsigned int* status = nullptr;
  if (cudaGetSymbolAddress(reinterpret_cast<void**>(&status), g_status) != cudaSuccess)
    return FA_ERR_LAUNCH;

  char* ws = static_cast<char*>(workspace);
  float* acc = reinterpret_cast<float*>(ws);
  CUtensorMap mdq;
  if (!encode_map_f32_acc(&mdq, acc, static_cast<int>(BH), L, d)) return FA_ERR_LAUNCH;
  float* nlse2 = reinterpret_cast<float*>(ws + w.acc_bytes);
  float* nds = reinterpret_cast<float*>(ws + w.acc_bytes + w.row_bytes);
  unsigned int* sched = reinterpret_cast<unsigned int*>(ws + w.acc_bytes + 2 * w.row_bytes);
  const int Lp = static_cast<int>(n_kv * 128);

  BwdArgs args;
  args.dk = static_cast<uint16_t*>(dk);
  args.dv = static_cast<uint16_t*>(dv);
  args.dq_acc = acc;
  args.nlse2 = nlse2;
  args.nds = nds;
  args.L = L;
  args.Lp = Lp;
  args.n_kv = static_cast<int>(n_kv);
  args.bh = static_cast<int>(BH);
  args.n_units = static_cast<int>(BH * n_kv);
  args.sched = sched;
  {
    // Heads per scheduling group: Q + dO (bf16) and the fp32 dQ accumulator
    // of a group within ~32 MB of L2.
    const int64_t head_bytes = static_cast<int64_t>(L) * d * 8;
    const int64_t g = (int64_t{32} << 20) / head_bytes;
    args.group_heads = static_cast<int>(g < 1 ? 1 : (g > BH ? BH : g));
  }
  args.scale_log2 = scale * 1.4426950408889634f;
  args.scale = scale;
  args.status = status;
  args.timeout_ns = g_timeout_ns;
  args.test_withhold_kv = g_test_withhold_q;

  BwdPreArgs pre;
  pre.o = static_cast<const uint16_t*>(o);
  pre.dout = static_cast<const uint16_t*>(dout);
  pre.lse = lse;
  pre.nlse2 = nlse2;
  pre.nds = nds;
  pre.dq_acc = acc;
  pre.sched = sched;
  pre.L = L;
  pre.Lp = Lp;
  pre.rows = BH * Lp;
  pre.scale = scale;

  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint16_t* dq16 = static_cast<uint16_t*>(dq);
  if (d == 64)
    return causal ? launch_bwd<64, true>(mq, mk, mv, mdo, mdq, args, pre, dq16, s, dev)
                  : launch_bwd<64, false>(mq, mk, mv, mdo, mdq, args, pre, dq16, s, dev);
  return causal ? launch_bwd<128, true>(mq, mk, mv, mdo, mdq, args, pre, dq16, s, dev)
                : launch_bwd<128, false>(mq, mk, mv, mdo, mdq, args, pre, dq16, s, dev);
}

int fa_quantize_fp8(const void* x, void* codes, float* scales, int B, int H, int L, int d,
                    fa_stream_t stream) {
  using namespace fa;
  if (!x || !codes || !scales || B < 1 || H < 1 || L < 1) return FA_ERR_INVALID_ARG;
  if (d != 64 && d != 128) return FA_ERR_UNSUPPORTED_D;
  const int64_t BH = static_cast<int64_t>(B) * H;
  const int64_t nb = (static_cast<int64_t>(L) + 127) / 128;
  if (BH * nb > 0x7fffffff) return FA_ERR_INVALID_ARG;
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scales, 4)) return FA_ERR_MISALIGNED;
  int dev = -1, major = 0, minor = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return FA_ERR_DEVICE;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
    return FA_ERR_DEVICE;
  if (major != 10 || minor != 3) return FA_ERR_DEVICE;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const dim3 grid(static_cast<unsigned>(BH * nb));
  const uint16_t* xs = static_cast<const uint16_t*>(x);
  uint8_t* cs = static_cast<uint8_t*>(codes);
  if (d == 64)
    fa_quantize_fp8_kernel<64><<<grid, QUANT_THREADS, 0, s>>>(xs, cs, scales, L, static_cast<int>(nb));
  else
    fa_quantize_fp8_kernel<128><<<grid, QUANT_THREADS, 0, s>>>(xs, cs, scales, L, static_cast<int>(nb));
  return cudaGetLastError() == cudaSuccess ? FA_OK : FA_ERR_LAUNCH;
}

int fa_fwd_fp8(const void* q8, const void* k8, const void* v, const float* q_scale,
               const float* k_scale, void* o, float* lse, int B, int H, int L, int d, float scale,
               int causal, fa_stream_t stream) {
  using namespace fa;
  if (!q_scale || !k_scale) return FA_ERR_INVALID_ARG;
  if (!aligned(q_scale, 4) || !aligned(k_scale, 4)) return FA_ERR_MISALIGNED;
  Prepared p;
  const int rc = prepare(q8, k8, v, o, lse, B, H, L, d, scale, causal, &p);
  if (rc != FA_OK) return rc;
  // Q and K are E4M3 codes: one-byte tensor maps in place of the bf16 ones.
  if (!encode_map_u8(&p.mq, q8, p.args.bh, L, d) || !encode_map_u8(&p.mk, k8, p.args.bh, L, d))
    return FA_ERR_LAUNCH;
  p.args.q_scale = q_scale;
  p.args.k_scale = k_scale;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (d == 64)
    return causal ? launch<64, true, false, true>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                  : launch<64, false, false, true>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
  return causal ? launch<128, true, false, true>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                : launch<128, false, false, true>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
}

size_t fa_fwd_host_workspace_bytes(int B, int H, int L, int d) {
  if (B < 1 || H < 1 || L < 1 || (d != 64 && d != 128)) return 0;
  const size_t n = static_cast<size_t>(B) * H * L * d * 2;  // bytes of one bf16 tensor
  return fa::align256(4 * n) + static_cast<size_t>(B) * H * L * 4;
}

int fa_fwd_host(const void* q, const void* k, const void* v, void* o, float* lse, int B, int H,
                int L, int d, float scale, int causal, void* workspace, size_t workspace_bytes,
                fa_stream_t stream) {
  using namespace fa;
  if (!q || !k || !v || !o || !lse || !workspace) return FA_ERR_INVALID_ARG;
  const size_t need = fa_fwd_host_workspace_bytes(B, H, L, d);
  if (need == 0) return (d != 64 && d != 128 && B >= 1 && H >= 1 && L >= 1)
                            ? FA_ERR_UNSUPPORTED_D : FA_ERR_INVALID_ARG;
  if (workspace_bytes < need) return FA_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return FA_ERR_MISALIGNED;
  const size_t n = static_cast<size_t>(B) * H * L * d * 2;
  const size_t nl = static_cast<size_t>(B) * H * L * 4;
  char* ws = static_cast<char*>(workspace);
  // device copies: Q, K, V, O back to back, then LSE
  char* dq = ws;
  char* dk = ws + n;
  char* dv = ws + 2 * n;
  char* dout = ws + 3 * n;
  float* dlse = reinterpret_cast<float*>(ws + align256(4 * n));
  // Validate every argument (with the device buffers) before any copy.
  Prepared p;
  int rc = prepare(dq, dk, dv, dout, dlse, B, H, L, d, scale, causal, &p);
  if (rc != FA_OK) return rc;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const char* hq = static_cast<const char*>(q);
  const char* hk = static_cast<const char*>(k);
  const char* hv = static_cast<const char*>(v);
  // inputs adjacent in host memory travel in one copy (the device copies are)
  if (hk == hq + n && hv == hk + n) {
    if (cudaMemcpyAsync(dq, hq, 3 * n, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  } else {
    if (cudaMemcpyAsync(dq, hq, n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dk, hk, n, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(dv, hv, n, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  if (d == 64)
    rc = causal ? launch<64, true, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                : launch<64, false, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
  else
    rc = causal ? launch<128, true, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev)
                : launch<128, false, false>(p.mq, p.mk, p.mv, p.args, 1, s, p.dev);
  if (rc != FA_OK) return rc;
  char* ho = static_cast<char*>(o);
  char* hl = reinterpret_cast<char*>(lse);
  if (hl == ho + n && reinterpret_cast<char*>(dlse) == dout + n) {
    if (cudaMemcpyAsync(ho, dout, n + nl, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  } else {
    if (cudaMemcpyAsync(ho, dout, n, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(hl, dlse, nl, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return FA_ERR_LAUNCH;
  }
  return FA_OK;
}

int fa_device_status(fa_stream_t stream, int clear) {
  using namespace fa;
  if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FA_ERR_LAUNCH;
  unsigned int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status, sizeof(v)) != cudaSuccess) return FA_ERR_LAUNCH;
  if (clear) {
    const unsigned int zero = 0;
    if (cudaMemcpyToSymbol(g_status, &zero, sizeof(zero)) != cudaSuccess) return FA_ERR_LAUNCH;
  }
  return v ? FA_ERR_TIMEOUT : FA_OK;
}

void fa_set_wait_timeout_ns(uint64_t ns) { fa::g_timeout_ns = ns < 1000 ? 1000 : ns; }

void fa_test_withhold_q_load(int enable) { fa::g_test_withhold_q = enable ? 1 : 0; }

const char* fa_status_string(int status) {
  switch (status) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED_D: return "unsupported head dimension (64 or 128)";
    case FA_ERR_MISALIGNED: return "misaligned pointer (q, k, v, o need 16 bytes; lse 4)";
    case FA_ERR_DEVICE: return "no usable sm_103 device";
    case FA_ERR_LAUNCH: return "CUDA launch or runtime error";
    case FA_ERR_TIMEOUT: return "a kernel wait timed out";
    default: return "unknown status";
  }
}

int fa_version(void) { return 300; }

}  // extern "C"
