// kernels.h -- internal launchers of libattn (not part of the C ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "common.cuh"

namespace attn {

// ---- tensor maps (host) ---------------------------------------------------
// A 3-D bf16 tensor map over [z][y][x] (x innermost, contiguous), with the
// 128-byte swizzle and zero fill outside the tensor.  box_x * 2 must be 128.
// Rows are ld elements apart (ld = 0: packed, ld = x; ld * 2 a multiple of 16).
bool make_tmap_bf16(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                    uint32_t box_x, uint32_t box_y, uint64_t ld = 0);
// A 3-D 8-bit tensor map over [z][y][x], 128-byte swizzle, zero fill outside
// the tensor (box_x must be 128; x a multiple of 16).
bool make_tmap_u8(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                  uint32_t box_x, uint32_t box_y);
// A 3-D fp32 tensor map over [z][y][x] for reduce-add tiles; with sw128 the
// shared-memory tile uses the 128-byte swizzle (box_x * 4 must then be 128).
bool make_tmap_f32(CUtensorMap* map, const void* base, uint64_t x, uint64_t y, uint64_t z,
                   uint32_t box_x, uint32_t box_y, bool sw128 = false);

KernelCtl default_ctl();

// Unique id of the CUDA context current on this thread (the runtime's
// primary context of the current device unless the caller made another one
// current); 0 if it cannot be read.  Device addresses of the library's
// file-scope __device__ arrays are cached per context under this id.
unsigned long long current_context_id();

// One block whose only wait has no arrival: records ATTN_ERR_DEVICE_TIMEOUT
// after timeout_ns and returns (attn_selftest_wait_timeout).
cudaError_t launch_wait_selftest(uint64_t timeout_ns, cudaStream_t st);

// Counts one kernel launch of the library (host side; attn_launch_count).
void note_launch();
unsigned long long launch_count();

// Block-sparse tile lists (built by launch_tile_lists in sparse.cu): for
// outer unit u, lists[u * stride + p], p < counts[u], are the inner tiles to
// visit in increasing order, each entry the tile index (low 16 bits) with one
// bit per member tile of the unit (bit 16 + m) for "kept for member m".
struct TileLists {
  const int* lists = nullptr;   // null: dense
  const int* counts = nullptr;
  int stride = 0;
};

// ---- fp32 SIMT path --------------------------------------------------------
// BH counts query heads (B * H); K, V (and dK, dV) hold BH / hm.group heads.
// bmask: block-sparse pattern, uint8 [ceil(n/128)][ceil(n/128)] (null: dense).
cudaError_t launch_fwd_f32(const float* Q, const float* K, const float* V, float* O, float* LSE,
                           int BH, const HeadMap& hm, const uint8_t* bmask, int n, int d,
                           float scale, int causal, cudaStream_t st);
cudaError_t launch_delta_f32(const float* O, const float* dO, float* Dv, int BH, int n, int d,
                             cudaStream_t st);
cudaError_t launch_bwd_dkdv_f32(const float* Q, const float* K, const float* V, const float* dO,
                                const float* LSE, const float* Dv, float* dK, float* dV, int BH,
                                const HeadMap& hm, const uint8_t* bmask, int n, int d, float scale,
                                int causal, cudaStream_t st);
cudaError_t launch_bwd_dq_f32(const float* Q, const float* K, const float* V, const float* dO,
                              const float* LSE, const float* Dv, float* dQ, int BH,
                              const HeadMap& hm, const uint8_t* bmask, int n, int d, float scale,
                              int causal, cudaStream_t st);

// ---- bf16 helpers ------------------------------------------------------------
cudaError_t launch_delta_bf16(const void* O, const void* dO, const float* LSE, float* Dv,
                              float* LSE2, float* dQacc, int BH, int n, int n_pad, int d,
                              cudaStream_t st);
cudaError_t launch_dq_convert(const float* acc, void* dQ, size_t elems, cudaStream_t st);

// ---- tensor-core kernels -------------------------------------------------------
// lda: row length of A in elements (0: packed); batches of A lda * rows apart.
int launch_gemm_bf16(const void* A, const void* B, void* C, int batch, int M, int N, int K,
                     bool a_kmajor, bool b_kmajor, bool c_f32, float alpha, const KernelCtl& ctl,
                     cudaStream_t st, int lda = 0);

// tl.lists != null: block-sparse (one key/value head per query head only).
int launch_fwd_tc(const void* Q, const void* K, const void* V, void* O, float* LSE, int BH,
                  const HeadMap& hm, const TileLists& tl, int n, int d, float scale, int causal,
                  const KernelCtl& ctl, cudaStream_t st);
// The forward's tiling for head dim d: a CTA owns query_tiles tiles of
// query_rows rows and walks KV tiles of kv_rows keys.
void fwd_tiling(int d, int* query_rows, int* query_tiles, int* kv_rows);

// Key-tile backward: dK, dV (and, with dQacc != nullptr, atomic dQ shares).
// One CTA per (key tile, key/value head, part of the group) walks the query
// tiles of the query heads of its part, so dK and dV sum over them in tensor
// memory.  gsplit = 1: one part, dK and dV stored as bf16.  gsplit > 1: each
// part adds its sums into the fp32 accumulators dKacc, dVacc (zeroed by the
// caller; dK already scaled), which the caller converts.
// tl.lists != null: block-sparse, each key tile walking its listed query
// tiles (one key/value head per query head only).
// dSt (d = 256, dense, one key/value head per query head, non-causal only):
// the dK CTAs also store dS^T in bf16, [BH][n keys][ld_ds queries], for dQ by
// a GEMM afterwards.
int launch_bwd_kv_tc(const void* Q, const void* K, const void* V, const void* dO,
                     const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                     float* dKacc, float* dVacc, int BH, const HeadMap& hm, int gsplit,
                     const TileLists& tl, int n, int n_pad, int d, float scale, int causal,
                     const KernelCtl& ctl, cudaStream_t st, void* dSt = nullptr, int ld_ds = 0);
// Tiling of the key-tile kernel for head dim d (key tiles of kv_rows keys,
// query tiles of query_rows).
void bwd_kv_tiling(int d, int* kv_rows, int* query_rows);
// Key-tile backward for d = 64 and d = 128, pipelined two query tiles deep
// (dQ shares reduced into dQacc with TMA bulk reduce-add when dQacc != nullptr).
int launch_bwd_kv64_tc(const void* Q, const void* K, const void* V, const void* dO,
                       const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                       float* dKacc, float* dVacc, int BH, const HeadMap& hm, int gsplit,
                       const TileLists& tl, int n, int n_pad, float scale, int causal,
                       const KernelCtl& ctl, cudaStream_t st);
int launch_bwd_kv128_tc(const void* Q, const void* K, const void* V, const void* dO,
                        const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                        float* dKacc, float* dVacc, int BH, const HeadMap& hm, int gsplit,
                        const TileLists& tl, int n, int n_pad, float scale, int causal,
                        const KernelCtl& ctl, cudaStream_t st);
// The key-tile backward with key tiles of key_rows keys (128, 64 or 32), for
// measuring how its memory traffic depends on the keys a CTA keeps on chip:
// each CTA still computes a 128-key tile but owns only its first key_rows
// keys.  Dense, one key/value head per query head.  d = 64 and 128 add dQ
// shares into dQacc (required); d = 256 takes none (dQacc must be null).
int launch_bwd_kv_study(const void* Q, const void* K, const void* V, const void* dO,
                        const float* LSE2, const float* Dv, float* dQacc, void* dK, void* dV,
                        int BH, int key_rows, int n, int n_pad, int d, float scale, int causal,
                        const KernelCtl& ctl, cudaStream_t st);
int launch_bwd_kv_study_d64_128(const void* Q, const void* K, const void* V, const void* dO,
                                const float* LSE2, const float* Dv, float* dQacc, void* dK,
                                void* dV, int BH, int key_rows, int n, int n_pad, int d,
                                float scale, int causal, const KernelCtl& ctl, cudaStream_t st);
// Query-tile backward: dQ with no atomics.
int launch_bwd_q_tc(const void* Q, const void* K, const void* V, const void* dO,
                    const float* LSE2, const float* Dv, void* dQ, int BH, const HeadMap& hm,
                    const TileLists& tl, int n, int n_pad, int d, float scale, int causal,
                    const KernelCtl& ctl, cudaStream_t st);
// Tiling of the query-tile dQ kernel (query tiles of query_rows, key tiles of kv_rows).
void bwd_q_tiling(int d, int* query_rows, int* kv_rows);

// FP8 (e4m3) forward for d = 128: Q, K [BH][n][128], Vt [BH][128][n] e4m3 bytes,
// O bf16 [BH][n][128], LSE fp32.  n must be a multiple of 16.
// descale_q/k/v: device arrays of BH floats, or null for 1.
int launch_fwd_fp8(const void* Q8, const void* K8, const void* Vt8, void* O, float* LSE, int BH,
                   int n, float scale, const float* descale_q, const float* descale_k,
                   const float* descale_v, int causal, const KernelCtl& ctl, cudaStream_t st);

// Per-head e4m3 quantisation of X bf16 [BH][n][128] into X8 ([BH][n][128],
// or [BH][128][n] when transpose) and descale [BH]; signs (128 floats of +-1)
// or null selects the Hadamard rotation.  partial: quant_fp8_workspace_bytes.
size_t quant_fp8_workspace_bytes(int BH, int n);
cudaError_t launch_quant_fp8(const void* X, void* X8, float* descale, int BH, int n, bool transpose,
                             const float* signs, float* partial, cudaStream_t st);

// ---- block-sparse tile lists (sparse.cu) ----------------------------------------------
size_t tile_lists_bytes(int n, int osz, int members, int isz);
cudaError_t launch_tile_lists(const uint8_t* mask, int n, int causal, bool outer_is_query, int osz,
                              int members, int isz, int* buf, cudaStream_t st);

// ---- materialise-P row kernels ----------------------------------------------------
cudaError_t launch_mat_softmax(const float* S, void* P, float* LSE, int BH, int n, float scale,
                               int causal, cudaStream_t st);
cudaError_t launch_mat_dsoftmax(const void* P, const float* dP, const float* Dv, void* dS, int BH,
                                int n, cudaStream_t st);

}  // namespace attn
