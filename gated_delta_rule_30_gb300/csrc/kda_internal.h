// kda_internal.h -- declarations shared by the library's translation units.
//
// Data flow of one kda_fwd call (all on the caller's stream):
//   1. schedule kernel: cu_seqlens (or B x T) -> per-sequence chunk offsets and
//      a table of 64-token chunks (start token, valid length); validates
//      cu_seqlens on the device.
//   2. chunk kernel (kda_prep.cu), one CTA per (chunk, head), fully parallel:
//      gate, in-chunk decays, the intra-chunk score matrices on tcgen05, the
//      unit-lower-triangular inverse, and the WY factors W, U on tcgen05.  It
//      writes one fixed-size record per (chunk, head) whose operand tiles are
//      already in the tcgen05 shared-memory layouts the next kernel uses.
//   3. recurrence kernel (kda_recur.cu), one CTA per (sequence, head, value
//      slice): keeps the fp32 state slice in TMEM, streams the records with
//      bulk copies and runs the sequential chunk-to-chunk update and outputs
//      on tcgen05.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "kda.h"

namespace kda {

constexpr int kChunk = 64;  // tokens per chunk
constexpr int kDim = 128;   // K = V = 128

// Per-(chunk, head) record written by the chunk kernel (byte offsets).
//   WQ : A operand [W ; scale*Qhat] of the state read-out, M = 128 rows (0..63 the
//        W rows of the chunk's tokens, 64..127 the decayed queries), K = 128 key
//        channels; MN-major, 8-row groups 2048 B apart, 8-channel groups 128 B apart.
//   KT : A operand Ktilde^T of the state update, M = 128 key channels, K = 64
//        tokens; K-major, 8-token groups 128 B apart, 8-channel groups 1024 B apart.
//   AQ : scale*Aqk as an unevaluated bf16 sum hi + lo (lo = bf16(x - hi)),
//        each the rows 64..127 of an M = 128, K = 64 token A operand; K-major,
//        8-token groups 128 B apart, 8-row groups 1024 B apart.  Rows 0..63 of
//        that operand are whatever lies
//        in the 8 KB before it: they only feed accumulator rows that are dead.
//   UT : U^T, [128 value channels][64 tokens] bf16 row-major.
//   GAM: chunk-end decay exp(G_last) per key channel, fp32 [128].
// The first kRecOperands bytes are copied verbatim into shared memory.
constexpr uint32_t kRecWQ = 0;
constexpr uint32_t kRecKT = 32768;
constexpr uint32_t kRecAQ = 49152;    // hi
constexpr uint32_t kRecAQL = 57344;   // lo
constexpr uint32_t kRecOperands = 65536;
constexpr uint32_t kRecUT = 65536;
constexpr uint32_t kRecGam = 81920;
constexpr uint32_t kRecBytes = 82432;

struct ChunkInfo {
    int32_t tok0;  // first token (row of the [total_tokens, H, 128] tensors)
    int32_t len;   // valid tokens, 1..64
};

// Workspace carve-up (all offsets 256-byte aligned).
struct Workspace {
    int32_t* flags;       // [0] = 1 when the schedule is valid
    int32_t* chunk_off;   // [N + 1] chunk prefix offsets per sequence
    ChunkInfo* info;      // [max_chunks]
    uint8_t* records;     // [max_chunks][H][kRecBytes]
};

struct Problem {
    const void* q;
    const void* k;
    const void* v;
    const void* g;
    const void* beta;
    float scale;
    void* out;
    const float* A_log;
    const float* dt_bias;
    float lower_bound;
    const void* h0;
    kda_dtype_t h0_dtype;
    void* hT;
    kda_dtype_t hT_dtype;
    const int32_t* cu;
    int32_t N;       // sequences
    int32_t B, T, H;
    int64_t total_tokens;
    int64_t max_chunks;
};

size_t workspace_bytes(int64_t max_chunks, int64_t N, int64_t H);
Workspace carve_workspace(void* base, int64_t max_chunks, int64_t N, int64_t H);

// Error reporting (thread-local message).
kda_status_t set_error(kda_status_t s, const char* msg);
kda_status_t cuda_error(cudaError_t e, const char* where);
void clear_error();

// Library status word on the current device (see kda_device_status).
int* device_status_ptr();
constexpr int kStatusDeviceInput = 1;
constexpr int kStatusTimeout = 2;

// Kernel launchers (kda_prep.cu, kda_recur.cu, kda_api.cu).
cudaError_t launch_schedule(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
cudaError_t launch_prep(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);
cudaError_t launch_recur(const Problem& p, const Workspace& ws, int* status, cudaStream_t st);

kda_status_t selftest_tcgen05(const void* a, const void* b, float* d, int N, int K,
                              cudaStream_t stream);

}  // namespace kda
