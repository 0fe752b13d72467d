// gift_encode_lowrank_noalloc: the rank-r GIFT encode for callers that cannot allocate
// device memory.
//
// gift_encode needs a caller-provided workspace for the projection partials, the scaled
// projection and the amax word.  Some callers cannot provide one: code that runs while a
// framework's caching allocator must not grow (inside a gradient hook or a communication
// callback), code that runs where cudaMalloc is not allowed to synchronise the device, and
// plain C programs that have no allocator of their own.  For them this entry point keeps
// that scratch in one fixed array in device memory that the library itself declares, so
// the call allocates nothing at all.
//
// The array (about 17 MiB) exists on every GPU that loads the library, for as long as the
// process lives.  All calls on a device share it: two calls whose work overlaps on the GPU
// (different streams without ordering between them) race on it and give wrong results, so
// order them on one stream or with events.  The amax word and the grid-barrier word are
// cleared by every call; the other scratch is fully overwritten before it is read.
//
// Set-up: the device address of the array is looked up once per device with
// cudaGetSymbolAddress, on the first call made with that device current.  Make that first
// call before any stream capture begins.
#include <mutex>

#include "kernels.cuh"

namespace {

constexpr int kNoAllocMaxRows = 4096;                        // d_out limit
constexpr int kNoAllocMaxCols = 16384;                       // d_in limit
constexpr size_t kNoAllocAmaxFloats = 64;                    // amax words and the barrier word, padded to 256 B
static_assert(gift::kEncodeBatchMax + 1 <= kNoAllocAmaxFloats, "the amax words and the barrier word fit the control block");
constexpr size_t kNoAllocPcFloats = (size_t)kNoAllocMaxRows * 32;
constexpr size_t kNoAllocPartFloats = (size_t)2 << 20;       // 8 MiB of projection partials
// tensor-core operand planes and counters (the lr_pipe_split_floats layout at the limits)
constexpr size_t kNoAllocSplitFloats = (size_t)64 * (kNoAllocMaxRows + kNoAllocMaxCols) + (size_t)48 * kNoAllocMaxCols +
                                       64;   // 8 MiB
constexpr size_t kNoAllocFloats = kNoAllocAmaxFloats + kNoAllocPcFloats + kNoAllocPartFloats + kNoAllocSplitFloats;

static __device__ __align__(256) float g_noalloc_scratch[kNoAllocFloats];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
float *g_scratch_addr[kMaxDevices] = {};

// Device address of the scratch array for the current device (looked up once per device).
cudaError_t scratch_address(int device, float **out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[device]) {
    void *p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[device] = static_cast<float *>(p);
  }
  *out = g_scratch_addr[device];
  return cudaSuccess;
}

}  // namespace

using namespace gift;

extern "C" gift_status gift_encode_lowrank_noalloc(gift_ctx *ctx, const gift_factor *f, const float *W, int d_out,
                                                   int d_in, gift_format fmt, const float *amax_in, void *codes,
                                                   float *scales, float *amax_out, int *d_status,
                                                   cudaStream_t stream) {
  if (!ctx || !f || !W || !codes || !scales || d_out <= 0 || d_in <= 0) return GIFT_ERR_INVALID_ARG;
  if (fmt != GIFT_FMT_E4M3 && fmt != GIFT_FMT_E5M2) return GIFT_ERR_INVALID_ARG;
  if (f->kind != GIFT_XF_LOWRANK || f->d_out != d_out || f->d_in != d_in) return GIFT_ERR_INVALID_ARG;
  if (!f->U || !f->mu || !f->sigma || f->rank < 1 || f->rank > kMaxRank || f->rank > d_in)
    return GIFT_ERR_INVALID_ARG;
  // size limits of the fixed scratch
  if (d_out > kNoAllocMaxRows || d_in > kNoAllocMaxCols) return GIFT_ERR_INVALID_ARG;
  if (lr_part_floats(ctx->sms, d_out, d_in) > kNoAllocPartFloats) return GIFT_ERR_INVALID_ARG;
  if (lr_pipe_split_floats(d_out, d_in) > kNoAllocSplitFloats) return GIFT_ERR_INVALID_ARG;
  int cur = -1;
  if (cudaGetDevice(&cur) != cudaSuccess || cur != ctx->device || cur < 0 || cur >= kMaxDevices)
    return GIFT_ERR_INVALID_ARG;
  float *base = nullptr;
  const cudaError_t se = scratch_address(cur, &base);
  if (se != cudaSuccess) {
    record_cuda_error(se);
    return GIFT_ERR_CUDA;
  }
  float *amax_ws = base;
  float *Pc = base + kNoAllocAmaxFloats;
  float *part = Pc + kNoAllocPcFloats;
  float *split = part + kNoAllocPartFloats;

  Launch L;
  L.stream = stream;
  L.sms = ctx->sms;
  L.status = d_status;
  float *planes = (d_in % 32 == 0) ? split : nullptr;
  LrApply a{};
  a.X = W;
  a.U = f->U;
  a.Pc = Pc;
  a.sigma = f->sigma;
  a.rank = f->rank;
  a.d_out = d_out;
  a.d_in = d_in;
  a.inverse = false;
  a.terms = 3;
  a.split = planes;
  if (planes) lr_u_planes(f->planes, split, d_out, d_in, &a.u_planes, &a.ut_planes);
  a.codes = static_cast<uint8_t *>(codes);
  a.scales = scales;
  a.amax_out = amax_out;
  a.amax_in = amax_in;
  a.amax_ws = amax_ws;
  a.grid_counter = reinterpret_cast<unsigned int *>(amax_ws + kEncodeBatchMax);
  if (lr_encode_batch_ok(L, a, LR_PACK_TENSOR) && lr_batch_part_floats(ctx->sms, d_out, d_in) <= kNoAllocPartFloats) {
    if (!f->planes && launch_lr_split_u_all(L, f->U, d_out, d_in, f->rank, 2, split) != cudaSuccess)
      return GIFT_ERR_CUDA;
    // the amax words and the grid-barrier word
    if (cudaMemsetAsync(amax_ws, 0, (kEncodeBatchMax + 1) * sizeof(float), stream) != cudaSuccess)
      return GIFT_ERR_CUDA;
    LrEncodeItem it{};
    it.X = W;
    it.codes = a.codes;
    it.scales = a.scales;
    it.amax_out = amax_out;
    it.amax_in = amax_in;
    if (launch_lr_encode_batch(L, LR_PACK_TENSOR, fmt, a, f->mu, part, lr_planes(split, d_out, d_in).pc, 1, &it) !=
        cudaSuccess)
      return GIFT_ERR_CUDA;
    return GIFT_OK;
  }
  if (lr_prepare_all(L, f->U, f->mu, f->sigma, f->rank, W, d_out, d_in, false, false, part, Pc, planes, f->planes) !=
      cudaSuccess)
    return GIFT_ERR_CUDA;
  if (!amax_in && cudaMemsetAsync(amax_ws, 0, sizeof(float), stream) != cudaSuccess) return GIFT_ERR_CUDA;
  if (lr_encode_fused_ok(L, a, LR_PACK_TENSOR)) {
    if (cudaMemsetAsync(a.grid_counter, 0, sizeof(unsigned int), stream) != cudaSuccess) return GIFT_ERR_CUDA;
    if (launch_lr_encode_fused(L, LR_PACK_TENSOR, fmt, a) != cudaSuccess) return GIFT_ERR_CUDA;
    return GIFT_OK;
  }
  if (!amax_in && launch_lr_apply(L, LR_AMAX, fmt, a) != cudaSuccess) return GIFT_ERR_CUDA;
  if (launch_lr_apply(L, LR_PACK_TENSOR, fmt, a) != cudaSuccess) return GIFT_ERR_CUDA;
  return GIFT_OK;
}
