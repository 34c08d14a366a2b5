// C ABI of libmoe.so: argument checking, allocation, and the fixed sequence of
// kernel launches on the caller's stream (no host synchronisation inside a
// forward call; all routing sizes stay on the device).
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>

#include "gdn.h"
#include "moe_internal.h"

using namespace moe;

struct moe_handle : public Handle {};

namespace {

thread_local char g_err[512] = "";

moe_status fail(moe_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

moe_status cuda_fail(cudaError_t e, const char* what) {
  if (e == cudaErrorMemoryAllocation)
    return fail(MOE_ERR_OOM, "%s: %s", what, cudaGetErrorString(e));
  return fail(MOE_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(call, what)                            \
  do {                                            \
    cudaError_t e_ = (call);                      \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

struct RouterPlan {
  int n, tiles, ks, m_units, units;
};

// K splits of the router GEMM: a function of d only (never of T), so that a
// token's logits -- and therefore its routing -- do not depend on how many
// tokens share the call or on the chunking.  Splits hold 8 K blocks (512).
int router_ksplit(int d) {
  const int kb = d / 64;
  int ks = 1;
  while (ks * 2 * 8 <= kb && kb % (ks * 2) == 0) ks *= 2;
  return ks;
}

// Token tiles of 128 rows, or of 64 when 128-row tiles leave SMs idle (each
// unit streams its share of the router weights from L2 whatever its width,
// so halving the tile pays only while the units do not exceed the SMs).
RouterPlan plan_router(const Handle* h, int T) {
  RouterPlan r;
  r.m_units = ceil_div(h->cfg.E, 256);
  r.ks = router_ksplit(h->cfg.d);
  r.n = T >= 128 ? 128 : ((T + 15) & ~15);
  if (r.n == 128 && ceil_div(T, 128) * r.m_units * r.ks < h->num_sms &&
      ceil_div(T, 64) * r.m_units * r.ks <= h->num_sms)
    r.n = 64;
  r.tiles = ceil_div(T, r.n);
  r.units = r.tiles * r.m_units * r.ks;
  return r;
}

int max_tiles_for(const Handle* h, int T) {
  const int k1 = h->cfg.k + (h->cfg.has_shared ? 1 : 0);
  return (int)((long long)T * k1 / kTileRows) + h->n_exp + 1;
}

void free_handle(Handle* h) {
  if (!h) return;
  void* ptrs[] = {h->pf_gu, h->pf_dn, h->pf_router, h->dc_gu, h->dc_dn, h->dc_router_t,
                  h->w_router, h->w_sg, h->dev_err, h->ws.logit_part, h->ws.logits,
                  h->ws.idx, h->ws.w, h->ws.sigma, h->ws.xp, h->ws.hist, h->ws.base,
                  h->ws.counts, h->ws.offsets, h->ws.perm, h->ws.slot, h->ws.dst, h->ws.wrow, h->ws.xrow, h->ws.xtok,
                  h->ws.tiles, h->ws.ntiles, h->ws.ticket, h->ws.H, h->ws.Y, h->ws.few,
                  h->ws.x_dev, h->ws.y_dev,
                  h->ws.bias_dev};
  for (void* p : ptrs)
    if (p) cudaFree(p);
  if (h->prof_ev) {
    for (int i = 0; i < Handle::kProfCalls * (Handle::kStagesTimed + 1); ++i)
      if (h->prof_ev[i]) cudaEventDestroy(h->prof_ev[i]);
    delete[] h->prof_ev;
  }
  delete static_cast<moe_handle*>(h);
}

template <typename T>
cudaError_t dalloc(T** p, size_t bytes) {
  return cudaMalloc(reinterpret_cast<void**>(p), bytes < 16 ? 16 : bytes);
}

moe_status validate_config(const moe_config* c) {
  if (!c) return fail(MOE_ERR_INVALID_ARG, "config is NULL");
  if (c->d < 256 || c->d % 256 != 0 || c->d > 16384)
    return fail(MOE_ERR_INVALID_ARG, "d=%d must be a multiple of 256 in [256, 16384]", c->d);
  if (c->E < 1 || c->E > kMaxE) return fail(MOE_ERR_INVALID_ARG, "E=%d not in [1, %d]", c->E, kMaxE);
  if (c->k < 1 || c->k > c->E || c->k > kMaxK)
    return fail(MOE_ERR_INVALID_ARG, "k=%d not in [1, min(E, %d)]", c->k, kMaxK);
  if (c->I < 128 || c->I % 128 != 0 || c->I > 8192)
    return fail(MOE_ERR_INVALID_ARG, "I=%d must be a multiple of 128 in [128, 8192]", c->I);
  if (c->group < 64 || c->group % 64 != 0 || c->d % c->group != 0 || c->I % c->group != 0)
    return fail(MOE_ERR_UNSUPPORTED, "group=%d: must be a multiple of 64 dividing d=%d and I=%d",
                c->group, c->d, c->I);
  if (c->scale_dtype != MOE_SCALE_F16 && c->scale_dtype != MOE_SCALE_BF16)
    return fail(MOE_ERR_INVALID_ARG, "scale_dtype=%d unknown", c->scale_dtype);
  if (c->max_tokens < 1 || c->max_tokens > (1 << 20))
    return fail(MOE_ERR_INVALID_ARG, "max_tokens=%d not in [1, 2^20]", c->max_tokens);
  if (c->has_shared != 0 && c->has_shared != 1)
    return fail(MOE_ERR_INVALID_ARG, "has_shared must be 0 or 1");
  if (c->layouts < 0 || c->layouts > 3) return fail(MOE_ERR_INVALID_ARG, "layouts bitmask");
  return MOE_OK;
}

moe_status alloc_all(Handle* h) {
  const moe_config& c = h->cfg;
  const int k1 = c.k + (c.has_shared ? 1 : 0);
  const long long T = c.max_tokens;
  if (h->layouts & MOE_LAYOUT_PREFILL) {
    CK(dalloc(&h->pf_gu, (size_t)h->n_exp * (c.I / 128) * (c.d / 64) * kCodeChunk), "alloc");
    CK(dalloc(&h->pf_dn, (size_t)h->n_exp * (c.d / 256) * (c.I / 64) * kCodeChunk), "alloc");
    CK(dalloc(&h->pf_router, (size_t)ceil_div(c.E, 256) * (c.d / 64) * kRouterChunk), "alloc");
  }
  if (h->layouts & MOE_LAYOUT_DECODE) {
    CK(dalloc(&h->dc_gu, (size_t)h->n_exp * 2 * c.I * (c.d / 2 + c.d / 16)), "alloc");
    CK(dalloc(&h->dc_dn, (size_t)h->n_exp * c.d * (c.I / 2 + c.I / 16)), "alloc");
    CK(dalloc(&h->dc_router_t, (size_t)c.d * decode_router_pitch(c.E) * 2), "alloc");
  }
  CK(dalloc(&h->w_router, (size_t)c.E * c.d * 2), "alloc");
  CK(dalloc(&h->w_sg, (size_t)c.d * 2), "alloc");
  CK(dalloc(&h->dev_err, 16), "alloc");
  CK(cudaMemset(h->dev_err, 0, 16), "memset");

  Workspace& w = h->ws;
  w.Tmax = c.max_tokens;
  w.part_elems = (size_t)router_ksplit(c.d) * T * c.E;
  const size_t dec_bytes = decode_scratch_bytes(h, 64) + 64 * 1024;
  size_t part_bytes = w.part_elems * 4;
  if (part_bytes < dec_bytes) part_bytes = dec_bytes;
  CK(dalloc(&w.logit_part, part_bytes), "alloc");
  const int nblk = ceil_div(T, kTokPerBlock);
  w.max_tiles = max_tiles_for(h, (int)T);
  CK(dalloc(&w.logits, (size_t)T * c.E * 4), "alloc");
  CK(dalloc(&w.idx, (size_t)T * c.k * 4), "alloc");
  CK(dalloc(&w.w, (size_t)T * c.k * 4), "alloc");
  CK(dalloc(&w.sigma, (size_t)T * 4), "alloc");
  CK(dalloc(&w.hist, (size_t)nblk * c.E * 4), "alloc");
  CK(dalloc(&w.base, (size_t)nblk * c.E * 4), "alloc");
  CK(dalloc(&w.counts, (size_t)c.E * 4), "alloc");
  CK(dalloc(&w.offsets, (size_t)(c.E + 1) * 4), "alloc");
  CK(dalloc(&w.perm, (size_t)T * k1 * 4), "alloc");
  CK(dalloc(&w.slot, (size_t)T * c.k * 4), "alloc");
  CK(dalloc(&w.dst, (size_t)T * k1 * 4), "alloc");
  CK(dalloc(&w.wrow, (size_t)T * k1 * 4), "alloc");
  CK(dalloc(&w.xrow, (size_t)T * k1 * 4), "alloc");
  CK(dalloc(&w.xtok, (size_t)T * 4), "alloc");
  CK(dalloc(&w.tiles, (size_t)w.max_tiles * sizeof(int4)), "alloc");
  CK(dalloc(&w.ntiles, 16), "alloc");
  CK(dalloc(&w.ticket, 16), "alloc");
  CK(cudaMemset(w.ticket, 0, 16), "memset");
  if (h->layouts & MOE_LAYOUT_PREFILL) {
    CK(dalloc(&w.xp, (size_t)T * c.d * 2), "alloc");
    CK(dalloc(&w.H, (size_t)T * k1 * c.I * 2), "alloc");
    CK(dalloc(&w.Y, (size_t)T * k1 * c.d * 2), "alloc");
    CK(make_tmap_16bit(&h->tm_h, w.H, T * k1, c.I, 16, false), "tensor map (H)");
  }
  // the few-token path (2..8 tokens on the decode layout), when its scratch is modest
  if ((h->layouts & MOE_LAYOUT_DECODE) && T >= 2 && few_scratch_bytes(h) <= ((size_t)256 << 20))
    CK(dalloc(&w.few, few_scratch_bytes(h)), "alloc");
  CK(dalloc(&w.x_dev, (size_t)T * c.d * 2), "alloc");
  CK(dalloc(&w.y_dev, (size_t)T * c.d * 2), "alloc");
  CK(dalloc(&w.bias_dev, (size_t)c.E * 4 * 64), "alloc");  // [64][E]: moe_decode_host
  return MOE_OK;
}

// Event i of the current profiled chunk (stage boundaries 0..kStagesTimed).
void prof_mark(Handle* h, int i, cudaStream_t st) {
  if (!h->prof || h->prof_calls >= Handle::kProfCalls) return;
  cudaEventRecord(h->prof_ev[h->prof_calls * (Handle::kStagesTimed + 1) + i], st);
}

// router GEMM -> fused routing (top-k, histogram, scan + tile map, scatter;
// with_xp: also the fp16 copy of the activations that the gate/up GEMM
// gathers its token rows from, and the shared gate)
moe_status run_routing(Handle* h, const uint16_t* x, const float* logits_in, int T,
                       const float* bias, bool with_xp, cudaStream_t st) {
  const moe_config& c = h->cfg;
  const float* part = logits_in;
  int ks = 1;
  if (!logits_in) {
    const RouterPlan rp = plan_router(h, T);
    MmaParams p{};
    p.kb_per_unit = (c.d / 64) / rp.ks;
    p.m_units = rp.m_units;
    p.units_per_tile = rp.m_units * rp.ks;
    p.nunits_host = rp.units;
    p.router_n = rp.n;
    p.rows_total = T;
    p.wA = h->pf_router;
    p.a_expert_stride = 0;
    p.a_unit_stride = (long long)(c.d / 64) * kRouterChunk;
    p.a_chunk = kRouterChunk;
    CK(make_tmap_16bit(&p.tmB, x, T, c.d, 16, true), "tensor map (x)");
    p.out_f32 = h->ws.logit_part;
    p.E = c.E;
    p.err = h->dev_err;
    const int grid = rp.units < h->num_sms ? rp.units : h->num_sms;
    prof_mark(h, 0, st);
    CK(launch_grouped_mma(MMA_ROUTER, p, grid, st), "router launch");
    part = h->ws.logit_part;
    ks = rp.ks;
  }
  prof_mark(h, 1, st);
  CK(launch_route(h, part, ks, T, bias, with_xp ? x : nullptr, st), "routing launch");
  return MOE_OK;
}

moe_status run_experts(Handle* h, const uint16_t* x, int T, uint16_t* y, cudaStream_t st) {
  const moe_config& c = h->cfg;
  Workspace& w = h->ws;
  const int mt = max_tiles_for(h, T);
  MmaParams p{};
  p.tiles = w.tiles;
  p.ntiles_dev = w.ntiles;
  p.err = h->dev_err;
  p.a_chunk = kCodeChunk;
  // gate/up + SwiGLU
  p.kb_per_unit = c.d / 64;
  p.m_units = c.I / 128;
  p.units_per_tile = p.m_units;
  p.wA = h->pf_gu;
  p.a_unit_stride = (long long)(c.d / 64) * kCodeChunk;
  p.a_expert_stride = p.a_unit_stride * (c.I / 128);
  p.xg = w.xp;
  p.perm = w.perm;
  p.row_xscale = w.xrow;
  p.xscaled = reinterpret_cast<const int*>(w.ticket + 1);
  p.ldx = c.d;
  p.H = w.H;
  p.ldh = c.I;
  long long units = (long long)mt * p.m_units;
  int grid = units < h->num_sms ? (int)units : h->num_sms;
  prof_mark(h, 2, st);
  CK(launch_grouped_mma(MMA_GATEUP, p, grid, st), "gate/up launch");
  // down projection + routing weight: one 128-row weight tile per unit
  p.kb_per_unit = c.I / 64;
  p.m_units = c.d / 128;
  p.units_per_tile = p.m_units;
  p.wA = h->pf_dn;
  p.a_unit_stride = (long long)(c.I / 64) * kCodeChunk;
  p.a_expert_stride = p.a_unit_stride * (c.d / 256);
  p.tmB = h->tm_h;
  p.Y = w.Y;
  p.ldy = c.d;
  p.dst_row = w.dst;
  p.row_scale = w.wrow;
  units = (long long)mt * p.m_units;
  grid = units < h->num_sms ? (int)units : h->num_sms;
  prof_mark(h, 3, st);
  CK(launch_grouped_mma(MMA_DOWN, p, grid, st), "down launch");
  prof_mark(h, 4, st);
  CK(launch_combine(h, T, y, st), "combine launch");
  prof_mark(h, 5, st);
  if (h->prof && h->prof_calls < Handle::kProfCalls) ++h->prof_calls;
  return MOE_OK;
}

moe_status check_handle(const moe_handle* h) {
  if (!h) return fail(MOE_ERR_INVALID_ARG, "handle is NULL");
  return MOE_OK;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of device memory";
    case MOE_ERR_DEVICE: return "device error";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_err; }

int moe_version(void) { return 1; }

moe_status moe_create(const moe_config* cfg, const moe_weights* w, void* stream,
                      moe_handle** out) {
  if (!out) return fail(MOE_ERR_INVALID_ARG, "out is NULL");
  *out = nullptr;
  moe_status s = validate_config(cfg);
  if (s != MOE_OK) return s;
  if (!w) return fail(MOE_ERR_INVALID_ARG, "weights is NULL");
  const void* need[] = {w->gu_codes, w->gu_scale, w->gu_bias, w->dn_codes,
                        w->dn_scale, w->dn_bias, w->w_router};
  for (const void* p : need)
    if (!p || !aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "weight pointer NULL or not 16-byte aligned");
  if (cfg->has_shared) {
    const void* sh[] = {w->sh_gu_codes, w->sh_gu_scale, w->sh_gu_bias, w->sh_dn_codes,
                        w->sh_dn_scale, w->sh_dn_bias, w->w_shared_gate};
    for (const void* p : sh)
      if (!p || !aligned(p, 16)) return fail(MOE_ERR_INVALID_ARG, "shared-expert pointer NULL or not 16-byte aligned");
  }
  moe_handle* h = new (std::nothrow) moe_handle();
  if (!h) return fail(MOE_ERR_OOM, "host allocation");
  h->cfg = *cfg;
  h->layouts = cfg->layouts ? cfg->layouts : (MOE_LAYOUT_PREFILL | MOE_LAYOUT_DECODE);
  if (const char* wl = getenv("MOE_WAIT_LIMIT_NS")) {
    const long long v = atoll(wl);
    if (v >= 100000 && v <= 10000000000ll) h->wait_ns = (uint64_t)v;
  }
  if (const char* uf = getenv("MOE_TEST_UNSET_FLAG")) h->test_unset_flag = atoi(uf) == 1;
  h->n_exp = cfg->E + (cfg->has_shared ? 1 : 0);
  cudaError_t e = cudaGetDevice(&h->device);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&h->num_sms, cudaDevAttrMultiProcessorCount, h->device);
  if (e != cudaSuccess) {
    free_handle(h);
    return cuda_fail(e, "device query");
  }
  int major = 0, minor = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, h->device);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, h->device);
  if (major != 10 || minor != 3) {
    free_handle(h);
    return fail(MOE_ERR_UNSUPPORTED, "device is sm_%d%d; this library is built for sm_103a", major, minor);
  }
  s = alloc_all(h);
  if (s != MOE_OK) {
    free_handle(h);
    return s;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  e = cudaMemsetAsync(h->dev_err, 0, 16, st);  // ordered before the repack's flag
  if (e == cudaSuccess) e = launch_repack(h, w, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  int rerr = 0;
  if (e == cudaSuccess) e = cudaMemcpy(&rerr, h->dev_err, sizeof(int), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) {
    free_handle(h);
    return cuda_fail(e, "repack");
  }
  if (rerr & kRepackScaleInexact) {
    free_handle(h);
    return fail(MOE_ERR_UNSUPPORTED,
                "a bf16 scale/bias has no exact fp16 value (magnitude above 65504, or below "
                "2^-17 with bits under 2^-24)");
  }
  h->last_stream = st;
  *out = h;
  return MOE_OK;
}

moe_status moe_destroy(moe_handle* h) {
  if (!h) return MOE_OK;
  cudaDeviceSynchronize();
  free_handle(h);
  return MOE_OK;
}

moe_status moe_route(moe_handle* h, const void* x, int T, const float* logit_bias,
                     float* logits_out, int32_t* idx, float* w, int32_t* counts,
                     int32_t* offsets, int32_t* perm, int32_t* slot, void* stream) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (!(h->layouts & MOE_LAYOUT_PREFILL))
    return fail(MOE_ERR_INVALID_ARG, "moe_route needs the PREFILL layout");
  if (T < 0 || T > h->cfg.max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d not in [0, max_tokens=%d]", T, h->cfg.max_tokens);
  if (T == 0) return MOE_OK;
  if (!x || !aligned(x, 16)) return fail(MOE_ERR_INVALID_ARG, "x NULL or not 16-byte aligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  s = run_routing(h, static_cast<const uint16_t*>(x), nullptr, T, logit_bias, false, st);
  if (s != MOE_OK) return s;
  const moe_config& c = h->cfg;
  const Workspace& ws = h->ws;
  if (logits_out) CK(cudaMemcpyAsync(logits_out, ws.logits, (size_t)T * c.E * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (idx) CK(cudaMemcpyAsync(idx, ws.idx, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (w) CK(cudaMemcpyAsync(w, ws.w, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (counts) CK(cudaMemcpyAsync(counts, ws.counts, (size_t)c.E * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (offsets) CK(cudaMemcpyAsync(offsets, ws.offsets, (size_t)(c.E + 1) * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (perm) CK(cudaMemcpyAsync(perm, ws.perm, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (slot) CK(cudaMemcpyAsync(slot, ws.slot, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  return MOE_OK;
}

moe_status moe_route_from_logits(moe_handle* h, const float* logits, int T,
                                 const float* logit_bias, int32_t* idx, float* w,
                                 int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* slot, void* stream) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (T < 0 || T > h->cfg.max_tokens)
    return fail(MOE_ERR_INVALID_ARG, "T=%d not in [0, max_tokens=%d]", T, h->cfg.max_tokens);
  if (T == 0) return MOE_OK;
  if (!logits || !aligned(logits, 4)) return fail(MOE_ERR_INVALID_ARG, "logits NULL or misaligned");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  s = run_routing(h, nullptr, logits, T, logit_bias, false, st);
  if (s != MOE_OK) return s;
  const moe_config& c = h->cfg;
  const Workspace& ws = h->ws;
  if (idx) CK(cudaMemcpyAsync(idx, ws.idx, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (w) CK(cudaMemcpyAsync(w, ws.w, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (counts) CK(cudaMemcpyAsync(counts, ws.counts, (size_t)c.E * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (offsets) CK(cudaMemcpyAsync(offsets, ws.offsets, (size_t)(c.E + 1) * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (perm) CK(cudaMemcpyAsync(perm, ws.perm, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  if (slot) CK(cudaMemcpyAsync(slot, ws.slot, (size_t)T * c.k * 4, cudaMemcpyDeviceToDevice, st), "copy");
  return MOE_OK;
}

// Largest T that moe_forward runs on the bandwidth path of the DECODE layout:
// T = 1 through the decode kernel, 2 <= T <= 8 through the few-token kernel
// (one launch streaming the union of the tokens' experts once; one decode
// pass per token where its scratch was not built).  Below it the tensor-core
// path's fixed costs (routing, tile map, K loops of whole weight tiles)
// exceed the weight streaming.  MOE_SMALL_T (1..8; 0 or 1: T = 1 only)
// overrides it.
static int small_t_limit() {
  static int lim = -1;
  if (lim < 0) {
    const char* e = getenv("MOE_SMALL_T");
    const int def = few_max_tokens();
    lim = e ? atoi(e) : def;
    if (lim < 1 || lim > def) lim = (e && atoi(e) == 0) ? 1 : def;
  }
  return lim;
}

moe_status moe_forward(moe_handle* h, const void* x, int T, const float* logit_bias, void* y,
                       void* stream) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (T == 0) return MOE_OK;
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16))
    return fail(MOE_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
  if (logit_bias && !aligned(logit_bias, 4)) return fail(MOE_ERR_INVALID_ARG, "bias misaligned");
  const moe_config& c = h->cfg;
  const char* xb = static_cast<const char*>(x);
  const char* yb = static_cast<const char*>(y);
  const size_t bytes = (size_t)T * c.d * 2;
  if (xb < yb + bytes && yb < xb + bytes) return fail(MOE_ERR_INVALID_ARG, "x and y overlap");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  h->last_stream = st;
  if (T <= small_t_limit() && (h->layouts & MOE_LAYOUT_DECODE)) {
    if (T >= 2 && few_supported(h, T)) {
      CK(launch_few(h, static_cast<const uint16_t*>(x), T, logit_bias, static_cast<uint16_t*>(y),
                    st),
         "few-token launch");
      return MOE_OK;
    }
    // one pass of the bandwidth-bound decode kernel per token (each token's
    // output depends on that token only)
    moe_handle* one[1] = {h};
    for (int t = 0; t < T; ++t)
      CK(launch_decode(reinterpret_cast<Handle* const*>(one), 1,
                       static_cast<const uint16_t*>(x) + (size_t)t * c.d, logit_bias, 1e-6f,
                       static_cast<uint16_t*>(y) + (size_t)t * c.d, nullptr, st),
         "decode launch");
    return MOE_OK;
  }
  if (!(h->layouts & MOE_LAYOUT_PREFILL))
    return fail(MOE_ERR_INVALID_ARG, "T > 1 needs the PREFILL layout");
  for (int t0 = 0; t0 < T; t0 += c.max_tokens) {
    const int tc = (T - t0) < c.max_tokens ? (T - t0) : c.max_tokens;
    const uint16_t* xc = static_cast<const uint16_t*>(x) + (size_t)t0 * c.d;
    uint16_t* yc = static_cast<uint16_t*>(y) + (size_t)t0 * c.d;
    s = run_routing(h, xc, nullptr, tc, logit_bias, true, st);
    if (s != MOE_OK) return s;
    s = run_experts(h, xc, tc, yc, st);
    if (s != MOE_OK) return s;
  }
  return MOE_OK;
}

moe_status moe_forward_host(moe_handle* h, const void* x_host, int T, const float* bias_host,
                            void* y_host, void* stream) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (T < 0) return fail(MOE_ERR_INVALID_ARG, "T=%d < 0", T);
  if (T == 0) return MOE_OK;
  if (!x_host || !y_host) return fail(MOE_ERR_INVALID_ARG, "x_host/y_host NULL");
  const moe_config& c = h->cfg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const float* bias = nullptr;
  if (bias_host) {
    CK(cudaMemcpyAsync(h->ws.bias_dev, bias_host, (size_t)c.E * 4, cudaMemcpyHostToDevice, st), "bias copy");
    bias = h->ws.bias_dev;
  }
  for (int t0 = 0; t0 < T; t0 += c.max_tokens) {
    const int tc = (T - t0) < c.max_tokens ? (T - t0) : c.max_tokens;
    const size_t bytes = (size_t)tc * c.d * 2;
    CK(cudaMemcpyAsync(h->ws.x_dev, static_cast<const char*>(x_host) + (size_t)t0 * c.d * 2,
                       bytes, cudaMemcpyHostToDevice, st), "x copy");
    s = moe_forward(h, h->ws.x_dev, tc, bias, h->ws.y_dev, stream);
    if (s != MOE_OK) return s;
    CK(cudaMemcpyAsync(static_cast<char*>(y_host) + (size_t)t0 * c.d * 2, h->ws.y_dev, bytes,
                       cudaMemcpyDeviceToHost, st), "y copy");
  }
  CK(cudaStreamSynchronize(st), "synchronise");
  return MOE_OK;
}

moe_status moe_decode(moe_handle* const* layers, int L, const void* x, const float* logit_bias,
                      float eps, void* y, const moe_decode_trace* trace, void* stream) {
  if (!layers || L < 1) return fail(MOE_ERR_INVALID_ARG, "need L >= 1 layers");
  if (!x || !y || !aligned(x, 16) || !aligned(y, 16))
    return fail(MOE_ERR_INVALID_ARG, "x/y NULL or not 16-byte aligned");
  if (!(eps >= 0.0f)) return fail(MOE_ERR_INVALID_ARG, "eps must be >= 0");
  const moe_handle* h0 = layers[0];
  if (!h0) return fail(MOE_ERR_INVALID_ARG, "layer 0 handle is NULL");
  for (int l = 0; l < L; ++l) {
    const moe_handle* h = layers[l];
    if (!h) return fail(MOE_ERR_INVALID_ARG, "layer %d handle is NULL", l);
    if (!(h->layouts & MOE_LAYOUT_DECODE))
      return fail(MOE_ERR_INVALID_ARG, "layer %d lacks the DECODE layout", l);
    if (h->cfg.d != h0->cfg.d || h->cfg.E != h0->cfg.E || h->cfg.k != h0->cfg.k ||
        h->cfg.I != h0->cfg.I || h->cfg.has_shared != h0->cfg.has_shared)
      return fail(MOE_ERR_INVALID_ARG, "layer %d shape differs from layer 0", l);
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const_cast<moe_handle*>(h0)->last_stream = st;
  CK(launch_decode(reinterpret_cast<Handle* const*>(layers), L, static_cast<const uint16_t*>(x),
                   logit_bias, eps, static_cast<uint16_t*>(y), trace, st),
     "decode launch");
  return MOE_OK;
}

moe_status moe_decode_host(moe_handle* const* layers, int L, const void* x_host,
                           const float* bias_host, float eps, void* y_host, void* stream) {
  if (!layers || L < 1 || !layers[0]) return fail(MOE_ERR_INVALID_ARG, "need L >= 1 layers");
  if (!x_host || !y_host) return fail(MOE_ERR_INVALID_ARG, "x_host/y_host NULL");
  if (bias_host && L > 64) return fail(MOE_ERR_INVALID_ARG, "bias_host needs L <= 64");
  moe_handle* h0 = layers[0];
  const moe_config& c = h0->cfg;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaMemcpyAsync(h0->ws.x_dev, x_host, (size_t)c.d * 2, cudaMemcpyHostToDevice, st), "x copy");
  const float* bias = nullptr;
  if (bias_host) {
    CK(cudaMemcpyAsync(h0->ws.bias_dev, bias_host, (size_t)L * c.E * 4, cudaMemcpyHostToDevice,
                       st), "bias copy");
    bias = h0->ws.bias_dev;
  }
  moe_status s = moe_decode(layers, L, h0->ws.x_dev, bias, eps, h0->ws.y_dev, nullptr, stream);
  if (s != MOE_OK) return s;
  CK(cudaMemcpyAsync(y_host, h0->ws.y_dev, (size_t)c.d * 2, cudaMemcpyDeviceToHost, st), "y copy");
  CK(cudaStreamSynchronize(st), "synchronise");
  return MOE_OK;
}

moe_status moe_profile_enable(moe_handle* h, int enable) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (enable && !h->prof_ev) {
    const int n = Handle::kProfCalls * (Handle::kStagesTimed + 1);
    h->prof_ev = new (std::nothrow) cudaEvent_t[n]();
    if (!h->prof_ev) return fail(MOE_ERR_OOM, "host allocation");
    for (int i = 0; i < n; ++i) CK(cudaEventCreate(&h->prof_ev[i]), "event create");
  }
  h->prof = enable != 0;
  h->prof_calls = 0;
  return MOE_OK;
}

moe_status moe_profile_read(moe_handle* h, float* ms, int n, int* calls) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (!ms || n < 0 || n > Handle::kStagesTimed) return fail(MOE_ERR_INVALID_ARG, "ms/n");
  CK(cudaDeviceSynchronize(), "synchronise");
  for (int i = 0; i < n; ++i) ms[i] = 0.f;
  const int S = Handle::kStagesTimed + 1;
  for (int c = 0; c < h->prof_calls; ++c) {
    for (int i = 0; i < n; ++i) {
      float t = 0.f;
      // a chunk routed from given logits has no router stage: its first event is unused
      if (cudaEventElapsedTime(&t, h->prof_ev[c * S + i], h->prof_ev[c * S + i + 1]) ==
          cudaSuccess)
        ms[i] += t;
      else
        cudaGetLastError();
    }
  }
  if (calls) *calls = h->prof_calls;
  h->prof_calls = 0;
  return MOE_OK;
}

moe_status moe_get_device_error(moe_handle* h, int* code) {
  moe_status s = check_handle(h);
  if (s != MOE_OK) return s;
  if (!code) return fail(MOE_ERR_INVALID_ARG, "code is NULL");
  CK(cudaStreamSynchronize(h->last_stream), "synchronise");
  int v = 0;
  CK(cudaMemcpy(&v, h->dev_err, 4, cudaMemcpyDeviceToHost), "read error word");
  CK(cudaMemset(h->dev_err, 0, 4), "clear error word");
  *code = v;
  return v ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status gdn_scan(const void* q, const void* k, const void* v, const float* g,
                    const float* beta, float scale, const int32_t* offsets, int N, int T,
                    int Hk, int Hv, int dk, int dv, const float* state_in, float* state_out,
                    void* o, void* stream) {
  if (T > 0 && (!q || !k || !v || !g || !beta || !o))
    return fail(MOE_ERR_INVALID_ARG, "NULL tensor");
  if (T < 0 || N < 1 || Hk < 1 || Hv < 1 || dk < 1 || dv < 1)
    return fail(MOE_ERR_INVALID_ARG, "bad size (T=%d N=%d Hk=%d Hv=%d dk=%d dv=%d)", T, N, Hk,
                Hv, dk, dv);
  if (Hv % Hk != 0) return fail(MOE_ERR_INVALID_ARG, "Hv=%d is not a multiple of Hk=%d", Hv, Hk);
  if (Hv > 65535 || N > 65535) return fail(MOE_ERR_INVALID_ARG, "Hv or N above 65535");
  if (!offsets && N != 1) return fail(MOE_ERR_INVALID_ARG, "offsets is NULL but N=%d", N);
  if (!(scale == scale) || scale > 3.0e38f || scale < -3.0e38f)
    return fail(MOE_ERR_INVALID_ARG, "scale is not finite");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) ||
      !aligned(state_in, 16) || !aligned(state_out, 16) || !aligned(g, 4) ||
      !aligned(beta, 4) || !aligned(offsets, 4))
    return fail(MOE_ERR_INVALID_ARG, "misaligned pointer");
  if (dk != kGdnDk) return fail(MOE_ERR_UNSUPPORTED, "dk=%d (supported: %d)", dk, kGdnDk);
  if (dv % kGdnRows != 0)
    return fail(MOE_ERR_UNSUPPORTED, "dv=%d is not a multiple of %d", dv, kGdnRows);
  if (T == 0 && !state_out) return MOE_OK;
  GdnParams p{};
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.g = g;
  p.beta = beta;
  p.offsets = offsets;
  p.state_in = state_in;
  p.state_out = state_out;
  p.o = static_cast<uint16_t*>(o);
  p.scale = scale;
  p.T = T;
  p.Hk = Hk;
  p.Hv = Hv;
  p.dv = dv;
  p.N = N;
  CK(launch_gdn_scan(p, static_cast<cudaStream_t>(stream)), "gdn_scan launch");
  return MOE_OK;
}

}  // extern "C"
