// Internal structures shared by the translation units of libmoe.so.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cstddef>
#include <cstdint>
#include <utility>

#include "moe.h"

namespace moe {

constexpr int kMaxE = 512;
constexpr int kMaxK = 16;
constexpr int kTokPerBlock = 32;  // tokens per block of the routing kernels
constexpr int kTileRows = 192;    // largest token tile of the grouped GEMMs (TMEM budget)
constexpr int kUnitRows = 256;    // weight rows per tensor-core work unit (2 x M=128)
constexpr int kCodeChunk = 9216;  // 256 rows x (32 B codes + 4 B scale/bias)
constexpr int kRouterChunk = 32768;  // 256 rows x 64 bf16, pre-swizzled
// device error word bit set by the repack when a bf16 scale/bias has no exact
// fp16 value (moe_create then refuses the weights; never seen by callers)
constexpr int kRepackScaleInexact = 1 << 30;

// Per-handle scratch, sized for cfg.max_tokens tokens.
struct Workspace {
  int Tmax = 0;
  size_t part_elems = 0;     // capacity of logit_part (floats)
  float* logit_part = nullptr;  // router partial sums [KS][T][E]
  float* logits = nullptr;      // [Tmax][E] final logits (bias included)
  int32_t* idx = nullptr;       // [Tmax][k]
  float* w = nullptr;           // [Tmax][k]
  float* sigma = nullptr;       // [Tmax]
  uint16_t* xp = nullptr;       // [Tmax][d] fp16 copy of the activations (gate/up B rows)
  int32_t* hist = nullptr;      // [nblk][E]
  int32_t* base = nullptr;      // [nblk][E]
  int32_t* counts = nullptr;    // [E]
  int32_t* offsets = nullptr;   // [E+1]
  int32_t* perm = nullptr;      // [Tmax*(k+1)] grouped row -> token
  int32_t* slot = nullptr;      // [Tmax][k]
  int32_t* dst = nullptr;       // [Tmax*(k+1)] grouped row -> contribution row
  float* wrow = nullptr;        // [Tmax*(k+1)] grouped row -> routing weight (times s^2)
  float* xrow = nullptr;        // [Tmax*(k+1)] grouped row -> activation scale s
  float* xtok = nullptr;        // [Tmax] activation scale s of each token
  int4* tiles = nullptr;        // [max_tiles] {expert, row0, nrows, npad}
  int32_t* ntiles = nullptr;    // [1]
  unsigned* ticket = nullptr;   // [4]: [2], [3] the routing launch's grid barrier (zero between calls);
                                // [1]: some token of the call has an activation scale s != 1
  uint16_t* H = nullptr;        // [Tmax*(k+1)][I] fp16 SwiGLU activations
  uint16_t* Y = nullptr;        // [Tmax*(k+1)][d] bf16 weighted contributions
  int max_tiles = 0;
  // few-token launches: abort flag, router sums, partials (null: not built)
  uint8_t* few = nullptr;
  // staging for moe_forward_host
  void* x_dev = nullptr;
  void* y_dev = nullptr;
  float* bias_dev = nullptr;
};

struct Handle {
  moe_config cfg{};
  int device = 0;
  int num_sms = 0;
  int layouts = 0;
  int n_exp = 0;  // E + has_shared (experts stored in the repacked arrays)
  // prefill layouts (tensor-core path)
  uint8_t* pf_gu = nullptr;      // [n_exp][I/128][d/64][kCodeChunk]
  uint8_t* pf_dn = nullptr;      // [n_exp][d/256][I/64][kCodeChunk]
  uint8_t* pf_router = nullptr;  // [ceil(E/256)][d/64][kRouterChunk]
  // decode layouts (bandwidth path)
  uint8_t* dc_gu = nullptr;      // [n_exp][I][gate codes | up codes | gate s,b | up s,b]
  uint8_t* dc_dn = nullptr;      // codes [n_exp][I/32][d][16 B], then s,b [n_exp][I/64][d]
  uint16_t* dc_router_t = nullptr;  // bf16 [d][Ep]: router transposed + w_sg column
  uint16_t* w_router = nullptr;  // bf16 [E][d]
  uint16_t* w_sg = nullptr;      // bf16 [d]
  Workspace ws;
  CUtensorMap tm_h;    // down B: H [Tmax*(k+1)][I], 16-row box
  // per-stage timing (moe_profile_enable)
  static constexpr int kStagesTimed = 5;
  static constexpr int kProfCalls = 4096;
  bool prof = false;
  int prof_calls = 0;
  cudaEvent_t* prof_ev = nullptr;  // [kProfCalls][kStagesTimed + 1]
  int* dev_err = nullptr;
  unsigned dec_epoch = 0;  // decode launches so far (tags the exchanged partials)
  // the decode kernels' waits on other CTAs give up after wait_ns (2 s;
  // MOE_WAIT_LIMIT_NS at moe_create); test_unset_flag (MOE_TEST_UNSET_FLAG=1
  // at moe_create, tests only) makes the decode kernel wait on a flag that
  // nothing sets, so that the give-up path runs
  uint64_t wait_ns = 2000000000ull;
  int test_unset_flag = 0;
  cudaStream_t last_stream = nullptr;
};

// Launches kern and returns that launch's own status (cudaGetLastError after a
// <<<>>> launch would also report, and clear, an error left by an earlier,
// unrelated launch).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                cudaStream_t st, Args&&... args) {
  cudaLaunchConfig_t c = {};
  c.gridDim = grid;
  c.blockDim = block;
  c.dynamicSmemBytes = smem;
  c.stream = st;
  return cudaLaunchKernelEx(&c, kern, std::forward<Args>(args)...);
}

// row pitch (elements) of the decode router layout: E router columns, the
// shared-gate column, zero padding to a 16-byte multiple
inline int decode_router_pitch(int E) { return ((E + 1) + 7) & ~7; }
// 32-bit scale/bias words per row of the decode down layout: I/64 groups,
// padded to a multiple of 4 (16-byte rows for bulk copies)

// ---- grouped tensor-core GEMM (grouped_mma.cu)
enum MmaMode { MMA_ROUTER = 0, MMA_GATEUP = 1, MMA_DOWN = 2 };

struct MmaParams {
  CUtensorMap tmB;      // B operand: 2-D map, 64 x rows box, 128-byte swizzle
  int kb_per_unit;      // 64-wide K blocks per work unit
  int m_units;          // 256-row weight units per tile
  int units_per_tile;   // m_units * ksplit
  int nunits_host;      // router only: total units
  const int4* tiles;    // grouped modes: device tile list
  const int32_t* ntiles_dev;
  int router_n;         // router: tokens per tile
  int rows_total;       // router: T
  // A operand
  const uint8_t* wA;
  long long a_expert_stride;  // bytes per expert
  long long a_unit_stride;    // bytes per 256-row unit
  int a_chunk;                // bytes per K block
  // B operand rows: router and down contiguous from row0 (16-row TMA tiles);
  // gate/up gathered by cp.async from row perm[row] of xg (fp16 [T][ldx])
  const uint16_t* xg;
  const int32_t* perm;
  int ldx;
  // epilogue
  float* out_f32;             // router partials [KS][T][E]
  int E;
  uint16_t* H;
  int ldh;
  uint16_t* Y;
  int ldy;
  const int32_t* dst_row;
  const float* row_scale;
  // gate/up: per grouped row, the power of two s that divided its fp16
  // activations (the epilogue undoes it); xscaled: nonzero when some token of
  // the call has s != 1 (otherwise the rows' scales are not read)
  const float* row_xscale;
  const int* xscaled;
  int* err;
};
cudaError_t launch_grouped_mma(int mode, const MmaParams& p, int grid, cudaStream_t st);
// 2-D tensor map over a row-major [rows][cols] 16-bit matrix, box {64, box_rows},
// 128-byte swizzle (the tensor-core operand layout), zero fill out of bounds
cudaError_t make_tmap_16bit(CUtensorMap* map, const void* base, long long rows, long long cols,
                            int box_rows, bool bf16);

// ---- routing (routing.cu)
// top-k, histogram, scan + tile map, scatter and (x non-null) the fp16 copy of
// the activations with the shared-expert gate, in one cooperative launch
cudaError_t launch_route(const Handle* h, const float* part, int KS, int T, const float* bias,
                         const uint16_t* x, cudaStream_t st);
cudaError_t launch_combine(const Handle* h, int T, uint16_t* y, cudaStream_t st);

// ---- repack (repack.cu)
cudaError_t launch_repack(Handle* h, const moe_weights* w, cudaStream_t st);

// ---- decode (decode.cu)
cudaError_t launch_decode(Handle* const* layers, int L, const uint16_t* x, const float* bias,
                          float eps, uint16_t* y, const moe_decode_trace* trace,
                          cudaStream_t st);
size_t decode_scratch_bytes(const Handle* h, int L);
// a few tokens (2..few_max_tokens()) of one layer in one launch (decode.cu):
// the union of the tokens' experts streamed once
size_t few_scratch_bytes(const Handle* h);
int few_max_tokens();
bool few_supported(const Handle* h, int T);
cudaError_t launch_few(Handle* h, const uint16_t* x, int T, const float* bias, uint16_t* y,
                       cudaStream_t st);

// Gated DeltaNet prefill scan (gdn_scan.cu).  Key width fixed at 128,
// value rows in blocks of 32; see include/gdn.h for the layouts.
struct GdnParams {
  const uint16_t* q;        // bf16 [T][Hk][128]
  const uint16_t* k;        // bf16 [T][Hk][128]
  const uint16_t* v;        // bf16 [T][Hv][dv]
  const float* g;           // [T][Hv] log of the gate
  const float* beta;        // [T][Hv]
  const int32_t* offsets;   // [N+1] or null (one sequence of T tokens)
  const float* state_in;    // [N][Hv][dv][128] or null (zero state)
  float* state_out;         // [N][Hv][dv][128] or null
  uint16_t* o;              // bf16 [T][Hv][dv]
  float scale;
  int T, Hk, Hv, dv, N;
};
constexpr int kGdnDk = 128;
constexpr int kGdnRows = 32;
cudaError_t launch_gdn_scan(const GdnParams& p, cudaStream_t st);

}  // namespace moe
