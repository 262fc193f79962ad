// df_pack.cu -- between the padded layout and the packed (unpadded) layout
// ("DisentangledFlash", section "Packed unpadded inference and training":
// pack_padded_with_info packs the valid tokens of a padded batch and returns
// the sequence offsets, unpack_packed scatters a packed result back; the
// packed kernels keep no [B, L, ...] workspace).
//
// A padded batch of B sequences of L positions with a padding mask [B, L]
// (0 = padding) becomes the valid positions of every sequence, in order,
// sequence after sequence; sequences without a valid position are dropped.
//   pack_info:  lens[b] = valid positions of sequence b; start[b] = exclusive
//               prefix of lens; cu_seqlens over the non-empty sequences;
//               info = {total tokens, longest sequence, non-empty sequences};
//               index[start[b] + k] = b * L + (position of the k-th valid one)
//   pack rows:  packed[t] = padded[index[t]]            t < total
//   unpack rows: padded[index[t]] = packed[t], every other row zero
// Every pass is a gather or a scatter of whole rows in 16-byte words; the
// only atomic is a shared-memory maximum (the longest sequence), whose result
// does not depend on order, so every output is deterministic.
#include <cstring>

#include "df_internal.h"

namespace df {
namespace {

constexpr int kScanThreads = 1024;

// lens[b] = number of non-zero bytes of mask[b * L .. b * L + L)
__global__ void seq_count_kernel(const uint8_t* __restrict__ mask, int L, int32_t* __restrict__ lens) {
    const int b = blockIdx.x;
    int c = 0;
    for (int l = threadIdx.x; l < L; l += blockDim.x) c += mask[(size_t)b * L + l] != 0;
    __shared__ int red[32];
    for (int o = 16; o > 0; o >>= 1) c += __shfl_xor_sync(0xffffffffu, c, o);
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = c;
    __syncthreads();
    if (threadIdx.x < 32) {
        int v = threadIdx.x < (int)(blockDim.x >> 5) ? red[threadIdx.x] : 0;
        for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (threadIdx.x == 0) lens[b] = v;
    }
}

// Block-wide inclusive scan of one int per thread (kScanThreads threads).
__device__ int block_scan_incl(int v, int* sh) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += u;
    }
    if (lane == 31) sh[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < (int)(blockDim.x >> 5) ? sh[lane] : 0;
        for (int o = 1; o < 32; o <<= 1) {
            const int u = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += u;
        }
        sh[lane] = w;
    }
    __syncthreads();
    const int r = v + (warp > 0 ? sh[warp - 1] : 0);
    __syncthreads();   // sh is reused by the next call
    return r;
}

// One block: start[b] (exclusive prefix of lens over all b), cu_seqlens over
// the non-empty sequences, info = {total, longest, non-empty count}.
__global__ void pack_scan_kernel(const int32_t* __restrict__ lens, int B, int32_t* __restrict__ start,
                                 int32_t* __restrict__ cu, int32_t* __restrict__ info) {
    __shared__ int sh[32];
    __shared__ int carry_tok, carry_seq, longest;
    if (threadIdx.x == 0) {
        carry_tok = carry_seq = longest = 0;
        cu[0] = 0;
    }
    __syncthreads();
    for (int b0 = 0; b0 < B; b0 += kScanThreads) {
        const int b = b0 + threadIdx.x;
        const int n = b < B ? lens[b] : 0;
        const int ne = n > 0 ? 1 : 0;
        const int tok_incl = block_scan_incl(n, sh);
        const int seq_incl = block_scan_incl(ne, sh);
        const int ct = carry_tok, cs = carry_seq;
        if (b < B) {
            start[b] = ct + tok_incl - n;
            if (ne) cu[cs + seq_incl] = ct + tok_incl;
            atomicMax(&longest, n);
        }
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) {
            carry_tok = ct + tok_incl;
            carry_seq = cs + seq_incl;
        }
        __syncthreads();
    }
    if (threadIdx.x == 0) {
        info[0] = carry_tok;
        info[1] = longest;
        info[2] = carry_seq;
    }
}

// One block per sequence: index[start[b] + k] = b * L + l for the k-th valid
// position l of sequence b (a block-wide scan of the mask, kScanThreads
// positions at a time).
__global__ void pack_index_kernel(const uint8_t* __restrict__ mask, int L, const int32_t* __restrict__ start,
                                  int32_t* __restrict__ index) {
    __shared__ int sh[32];
    __shared__ int carry;
    const int b = blockIdx.x;
    if (threadIdx.x == 0) carry = 0;
    __syncthreads();
    const int s0 = start[b];
    for (int l0 = 0; l0 < L; l0 += kScanThreads) {
        const int l = l0 + threadIdx.x;
        const int v = (l < L && mask[(size_t)b * L + l] != 0) ? 1 : 0;
        const int incl = block_scan_incl(v, sh);
        const int c = carry;
        if (v) index[s0 + c + incl - 1] = b * L + l;
        __syncthreads();
        if (threadIdx.x == kScanThreads - 1) carry = c + incl;
        __syncthreads();
    }
}

// out[t] = in[index[t]] for t < info[0] (rows of `words` 16-byte words); an
// index outside the input's in_rows rows (not from the matching pack_info)
// gives a zero row instead of a read out of bounds
__global__ void gather_rows_kernel(const uint4* __restrict__ in, long in_rows, const int32_t* __restrict__ index,
                                   const int32_t* __restrict__ info, long max_rows, int words,
                                   uint4* __restrict__ out) {
    const long total = info[0] < max_rows ? info[0] : max_rows;
    const long n = total * words;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const long t = x / words, w = x % words;
        const long r = index[t];
        out[x] = (r >= 0 && r < in_rows) ? in[r * words + w] : make_uint4(0u, 0u, 0u, 0u);
    }
}

// out[index[t]] = in[t] for t < info[0]; an index outside the output's
// out_rows rows is skipped
__global__ void scatter_rows_kernel(const uint4* __restrict__ in, const int32_t* __restrict__ index,
                                    const int32_t* __restrict__ info, long max_rows, int words,
                                    uint4* __restrict__ out, long out_rows) {
    const long total = info[0] < max_rows ? info[0] : max_rows;
    const long n = total * words;
    for (long x = (long)blockIdx.x * blockDim.x + threadIdx.x; x < n; x += (long)gridDim.x * blockDim.x) {
        const long t = x / words, w = x % words;
        const long r = index[t];
        if (r >= 0 && r < out_rows) out[r * words + w] = in[x];
    }
}

int grid_for(long n) {
    long blocks = (n + 255) / 256;
    if (blocks > 152L * 32) blocks = 152L * 32;
    return (int)(blocks < 1 ? 1 : blocks);
}

}  // namespace
}  // namespace df

using namespace df;

namespace {
bool al16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
bool al4(const void* p) { return ((uintptr_t)p & 3u) == 0; }
}  // namespace

extern "C" {

size_t df_pack_workspace_size(int32_t B) { return B < 1 ? 0 : (size_t)2 * sizeof(int32_t) * (size_t)B; }

df_status df_pack_info(const uint8_t* mask, int32_t B, int32_t L, int32_t* cu_seqlens, int32_t* index,
                       int32_t* info, void* workspace, size_t workspace_bytes, df_stream_t stream) {
    if (!mask || !cu_seqlens || !index || !info || B < 1 || L < 1) return DF_ERR_INVALID_ARG;
    if ((long long)B * L >= (1ll << 31)) return DF_ERR_UNSUPPORTED;
    if (!al4(cu_seqlens) || !al4(index) || !al4(info)) return DF_ERR_INVALID_ARG;
    if (!workspace || !al4(workspace) || workspace_bytes < df_pack_workspace_size(B)) return DF_ERR_WORKSPACE;
    cudaStream_t st = (cudaStream_t)stream;
    int32_t* lens = (int32_t*)workspace;
    int32_t* start = lens + B;
    seq_count_kernel<<<B, 256, 0, st>>>(mask, L, lens);
    pack_scan_kernel<<<1, kScanThreads, 0, st>>>(lens, B, start, cu_seqlens, info);
    pack_index_kernel<<<B, kScanThreads, 0, st>>>(mask, L, start, index);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

df_status df_pack_rows(const void* padded, int32_t padded_rows, const int32_t* index, const int32_t* info,
                       int32_t max_rows, size_t row_bytes, void* packed, df_stream_t stream) {
    if (!padded || !index || !info || !packed || max_rows < 1 || padded_rows < 1) return DF_ERR_INVALID_ARG;
    if (row_bytes == 0 || row_bytes % 16 || !al16(padded) || !al16(packed) || !al4(index) || !al4(info))
        return DF_ERR_INVALID_ARG;
    const int words = (int)(row_bytes / 16);
    gather_rows_kernel<<<grid_for((long)max_rows * words), 256, 0, (cudaStream_t)stream>>>(
        (const uint4*)padded, padded_rows, index, info, max_rows, words, (uint4*)packed);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

df_status df_unpack_rows(const void* packed, const int32_t* index, const int32_t* info, int32_t max_rows,
                         size_t row_bytes, int32_t padded_rows, void* padded, df_stream_t stream) {
    if (!padded || !index || !info || !packed || max_rows < 1 || padded_rows < 1) return DF_ERR_INVALID_ARG;
    if (row_bytes == 0 || row_bytes % 16 || !al16(padded) || !al16(packed) || !al4(index) || !al4(info))
        return DF_ERR_INVALID_ARG;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaMemsetAsync(padded, 0, row_bytes * (size_t)padded_rows, st) != cudaSuccess) return DF_ERR_CUDA;
    const int words = (int)(row_bytes / 16);
    scatter_rows_kernel<<<grid_for((long)max_rows * words), 256, 0, st>>>((const uint4*)packed, index, info,
                                                                          max_rows, words, (uint4*)padded,
                                                                          padded_rows);
    return cudaGetLastError() == cudaSuccess ? DF_OK : DF_ERR_CUDA;
}

}  // extern "C"
