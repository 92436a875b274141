// Plain fp64 CPU oracle for paged Multi-head Latent Attention (MLA) decode.
//
// TEST INFRASTRUCTURE ONLY. Nothing on the product path may call, link or
// load this file: only the tests, the smoke check and the benchmark's CPU
// baseline leg use it. It shares no code, header, table or constant with the
// CUDA library, and includes nothing from it.
//
// What is computed (the plain definition; the GPU kernels reach the same
// result up to rounding order):
//   For every request b and query head h, with L = seq_lens[b]:
//   1. gather   row_t = kv_cache[block_table[b][t / bs]][t % bs][0:576],
//               t = 0..L-1 (bf16 -> double is exact);
//   2. score    s_t = sm_scale * ( sum_{d<512} q_nope[b,h,d] * row_t[d]
//                                + sum_{d<64}  q_pe[b,h,d]   * row_t[512+d] );
//   3. softmax  m = max_t s_t, Z = sum_t exp(s_t - m), lse = m + ln Z;
//   4. output   out[b,h,j] = sum_t exp(s_t - m) / Z * row_t[j], j < 512
//               (V is the first 512 latent columns of the same row).
// Sources: "SM100 Cutlass MLA decode with unrestricted num_heads (< 128) for
// DeepSeek TP" (vLLM PR #20769), bot summary: split-KV partial results plus a
// reduction kernel that combines them; "[Kernel] Flashinfer MLA (trtllm-gen)
// decode kernel integration" (vLLM PR #21078), E2E Benchmark: paged latent
// cache served with --block-size 32. The latent row layout (512 c_kv then
// 64 k_pe, V = c_kv) and the natural-log LSE are the readings written down in
// the design notes; the pages print neither formulas nor tensor shapes.
//
// FP8 latent cache (oracle_mla_decode_fp8): each cached element is one byte
// in the OCP 8-bit E4M3 format and stands for kv_scale * e4m3(byte); step 1
// then reads that product, everything after it is unchanged. The pages name
// only an "fp8" KV cache ("[Kernel][DSV4.1] Fuse MXFP8 wo_b GEMM with
// sequence-parallel reduce-scatter" (vLLM PR #57428), serving command with
// --kv-cache-dtype fp8; "Support DS conv-state layout in fused KDA decode
// kernel" (vLLM PR #53396), E2E setup with an FP8 KV cache); the E4M3 format
// and one per-tensor scale are the readings taken there.
//
// Edge conventions: L = 0 gives out = 0 and lse = -inf. A block id outside
// [0, num_blocks) makes the call return ORACLE_ERR_BAD_BLOCK.
//
// Also here, each as its own routine so tests can pin one against another:
//   - oracle_mla_partial / oracle_mla_combine: the split-KV partial result of
//     a token range and the log-sum-exp merge of several partials;
//   - oracle_mla_decode_bruteforce: an independent second path (long double,
//     dense K materialised, exp without max subtraction) for tiny inputs.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <limits>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

constexpr int kDc = 512;              // latent c_kv columns (= V width)
constexpr int kDr = 64;               // rope k_pe columns
constexpr int kD = kDc + kDr;         // 576 columns per cached token row

constexpr int ORACLE_OK = 0;
constexpr int ORACLE_ERR_ARG = 1;
constexpr int ORACLE_ERR_BAD_BLOCK = 2;

// bf16 bit pattern -> double. bf16 is the top half of an IEEE binary32, so
// the widening is exact.
inline double bf16_to_double(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof(f));
  return static_cast<double>(f);
}

// OCP 8-bit floating point, E4M3 variant: bit 7 sign, bits 6..3 exponent
// with bias 7, bits 2..0 mantissa. Exponent field 0 holds the subnormals
// (mantissa / 8) * 2^-6; S.1111.111 is NaN; there are no infinities, so
// S.1111.110 = +-448 is the largest finite value.
double e4m3_to_double(uint8_t byte) {
  const int sign = byte >> 7;
  const int e = (byte >> 3) & 0xF;
  const int m = byte & 0x7;
  if (e == 0xF && m == 0x7) return std::numeric_limits<double>::quiet_NaN();
  const double mag = e == 0 ? std::ldexp(m / 8.0, -6) : std::ldexp(1.0 + m / 8.0, e - 7);
  return sign ? -mag : mag;
}

struct Inputs {
  int B, H;
  const uint16_t* q_nope;     // [B, H, 512]
  const uint16_t* q_pe;       // [B, H, 64]
  const uint16_t* kv_cache;   // [num_blocks, block_size, 576] bf16, or nullptr when kv_fp8 is set
  int64_t num_blocks;
  int block_size;
  const int32_t* block_table; // [B, max_blocks]
  int max_blocks;
  const int32_t* seq_lens;    // [B]
  double sm_scale;
  const uint8_t* kv_fp8 = nullptr;   // [num_blocks, block_size, 576] E4M3 bytes
  double kv_scale = 1.0;             // value = kv_scale * e4m3(byte)
};

// One gathered cache row (bf16 or FP8). values(dst, n) writes the values of
// its first n columns as doubles: the element type is decided once per row.
struct Row {
  const uint16_t* b16 = nullptr;
  const uint8_t* f8 = nullptr;
  double scale = 1.0;
  bool valid() const { return b16 != nullptr || f8 != nullptr; }
  void values(double* dst, int n) const {
    if (f8 != nullptr)
      for (int d = 0; d < n; ++d) dst[d] = scale * e4m3_to_double(f8[d]);
    else
      for (int d = 0; d < n; ++d) dst[d] = bf16_to_double(b16[d]);
  }
};

// Step 1: cached row t of request b (invalid for a block id out of range).
Row gather_row(const Inputs& in, int b, int64_t t) {
  const int64_t page = t / in.block_size;
  const int64_t slot = t % in.block_size;
  const int32_t blk = in.block_table[static_cast<int64_t>(b) * in.max_blocks + page];
  Row r;
  if (blk < 0 || blk >= in.num_blocks) return r;
  const int64_t off = (static_cast<int64_t>(blk) * in.block_size + slot) * kD;
  if (in.kv_fp8 != nullptr) {
    r.f8 = in.kv_fp8 + off;
    r.scale = in.kv_scale;
  } else {
    r.b16 = in.kv_cache + off;
  }
  return r;
}

// Step 2 for one token: the scaled score of head (b, h) against row.
double score(const Inputs& in, int b, int h, const Row& row) {
  const uint16_t* qn = in.q_nope + (static_cast<int64_t>(b) * in.H + h) * kDc;
  const uint16_t* qp = in.q_pe + (static_cast<int64_t>(b) * in.H + h) * kDr;
  double k[kD];
  row.values(k, kD);
  double acc = 0.0;
  for (int d = 0; d < kDc; ++d) acc += bf16_to_double(qn[d]) * k[d];
  for (int d = 0; d < kDr; ++d) acc += bf16_to_double(qp[d]) * k[kDc + d];
  return in.sm_scale * acc;
}

// Steps 1-4 over the listed tokens of request b for head h (each entry
// attended once, in any order). Writes the normalised output (out[512]) and
// the log-sum-exp of the list. An empty list gives zeros and -inf.
int attend_tokens(const Inputs& in, int b, int h, const std::vector<int64_t>& tokens,
                  double* out, double* lse) {
  for (int j = 0; j < kDc; ++j) out[j] = 0.0;
  if (tokens.empty()) {
    *lse = -std::numeric_limits<double>::infinity();
    return ORACLE_OK;
  }
  std::vector<double> s(tokens.size());
  std::vector<Row> rows(tokens.size());
  double m = -std::numeric_limits<double>::infinity();
  for (size_t i = 0; i < tokens.size(); ++i) {
    const Row row = gather_row(in, b, tokens[i]);
    if (!row.valid()) return ORACLE_ERR_BAD_BLOCK;
    rows[i] = row;
    s[i] = score(in, b, h, row);
    if (s[i] > m) m = s[i];
  }
  double z = 0.0;
  for (size_t i = 0; i < s.size(); ++i) {
    const double w = std::exp(s[i] - m);
    z += w;
    double v[kDc];
    rows[i].values(v, kDc);
    for (int j = 0; j < kDc; ++j) out[j] += w * v[j];
  }
  for (int j = 0; j < kDc; ++j) out[j] /= z;
  *lse = m + std::log(z);
  return ORACLE_OK;
}

// The same over the token range [t0, t1).
int attend_range(const Inputs& in, int b, int h, int64_t t0, int64_t t1,
                 double* out, double* lse) {
  std::vector<int64_t> tokens;
  for (int64_t t = t0; t < t1; ++t) tokens.push_back(t);
  return attend_tokens(in, b, h, tokens, out, lse);
}

bool valid_shape(const Inputs& in) {
  if (in.B < 0 || in.H < 1 || in.block_size < 1 || in.max_blocks < 0 || in.num_blocks < 0)
    return false;
  for (int b = 0; b < in.B; ++b) {
    if (in.seq_lens[b] < 0) return false;
    if (static_cast<int64_t>(in.seq_lens[b]) >
        static_cast<int64_t>(in.max_blocks) * in.block_size)
      return false;
  }
  return true;
}

int set_threads(int n_threads) {
#ifdef _OPENMP
  if (n_threads > 0) omp_set_num_threads(n_threads);
  return omp_get_max_threads();
#else
  (void)n_threads;
  return 1;
#endif
}

// Every query row of a decode whose requests carry q_len query tokens each:
// in.H counts q_len * heads rows per request, row j * heads + h, and token j
// attends to the first L - q_len + 1 + j cached tokens (all L for q_len = 1).
int decode_causal(const Inputs& in, int q_len, double* out, double* lse, int n_threads) {
  if (!valid_shape(in)) return ORACLE_ERR_ARG;
  const int heads = in.H / q_len;
  for (int b = 0; b < in.B; ++b)
    if (in.seq_lens[b] != 0 && in.seq_lens[b] < q_len) return ORACLE_ERR_ARG;
  set_threads(n_threads);
  const int64_t n = static_cast<int64_t>(in.B) * in.H;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    const int b = static_cast<int>(r / in.H);
    const int row = static_cast<int>(r % in.H);   // j * heads + h
    const int j = row / heads;
    const int64_t L = in.seq_lens[b];
    const int64_t Lj = L == 0 ? 0 : L - q_len + 1 + j;
    const int rc = attend_range(in, b, row, 0, Lj, out + r * kDc, lse + r);
    if (rc != ORACLE_OK) {
#pragma omp critical
      status = rc;
    }
  }
  return status;
}

}  // namespace

extern "C" {

// Number of OpenMP threads the oracle will use after applying n_threads
// (n_threads <= 0 keeps the runtime default).
int oracle_num_threads(int n_threads) { return set_threads(n_threads); }

// Full decode for a chosen list of (b, h) rows: out_rows[n_rows, 512],
// lse_rows[n_rows]. Rows are independent, so this is also the whole decode
// when the list holds every (b, h).
int oracle_mla_decode_rows(int B, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                           const uint16_t* kv_cache, int64_t num_blocks, int block_size,
                           const int32_t* block_table, int max_blocks,
                           const int32_t* seq_lens, double sm_scale, int64_t n_rows,
                           const int32_t* row_b, const int32_t* row_h, double* out_rows,
                           double* lse_rows, int n_threads) {
  Inputs in{B, H, q_nope, q_pe, kv_cache, num_blocks, block_size,
            block_table, max_blocks, seq_lens, sm_scale};
  if (!valid_shape(in)) return ORACLE_ERR_ARG;
  for (int64_t r = 0; r < n_rows; ++r)
    if (row_b[r] < 0 || row_b[r] >= B || row_h[r] < 0 || row_h[r] >= H) return ORACLE_ERR_ARG;
  set_threads(n_threads);
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n_rows; ++r) {
    const int b = row_b[r];
    const int rc = attend_range(in, b, row_h[r], 0, seq_lens[b], out_rows + r * kDc,
                                lse_rows + r);
    if (rc != ORACLE_OK) {
#pragma omp critical
      status = rc;
    }
  }
  return status;
}

// Full decode over every (b, h): out[B, H, 512], lse[B, H].
int oracle_mla_decode(int B, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                      const uint16_t* kv_cache, int64_t num_blocks, int block_size,
                      const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                      double sm_scale, double* out, double* lse, int n_threads) {
  if (B < 0 || H < 1) return ORACLE_ERR_ARG;
  const int64_t n = static_cast<int64_t>(B) * H;
  std::vector<int32_t> rb(static_cast<size_t>(n)), rh(static_cast<size_t>(n));
  for (int64_t i = 0; i < n; ++i) {
    rb[i] = static_cast<int32_t>(i / H);
    rh[i] = static_cast<int32_t>(i % H);
  }
  return oracle_mla_decode_rows(B, H, q_nope, q_pe, kv_cache, num_blocks, block_size,
                                block_table, max_blocks, seq_lens, sm_scale, n, rb.data(),
                                rh.data(), out, lse, n_threads);
}

// Multi-token decode (speculative decoding: q_len new tokens per request).
// q_nope [B, q_len, H, 512], q_pe [B, q_len, H, 64]; the request's length L
// counts the q_len new tokens, which are its last q_len tokens, so query
// token j (0-based) attends causally to tokens t < L - q_len + 1 + j.
// Writes out[B, q_len, H, 512] and lse[B, q_len, H]. Requires L == 0 (all
// rows empty: out = 0, lse = -inf) or L >= q_len. The causal rule is the
// reading taken where the pages only name speculative decoding.
int oracle_mla_decode_multi(int B, int q_len, int H, const uint16_t* q_nope,
                            const uint16_t* q_pe, const uint16_t* kv_cache, int64_t num_blocks,
                            int block_size, const int32_t* block_table, int max_blocks,
                            const int32_t* seq_lens, double sm_scale, double* out, double* lse,
                            int n_threads) {
  if (B < 0 || H < 1 || q_len < 1) return ORACLE_ERR_ARG;
  // The request's q_len x H query rows, row j * H + h, share its cache.
  Inputs in{B, q_len * H, q_nope, q_pe, kv_cache, num_blocks, block_size,
            block_table, max_blocks, seq_lens, sm_scale};
  return decode_causal(in, q_len, out, lse, n_threads);
}

// The same decode over an FP8 latent cache: kv_fp8 holds E4M3 bytes
// [num_blocks, block_size, 576] and element (blk, slot, d) stands for
// kv_scale * e4m3(kv_fp8[blk, slot, d]). q_len = 1 is the ordinary decode
// (q [B, H, ...], out [B, H, 512], lse [B, H]); q_len > 1 follows the
// causal rule of oracle_mla_decode_multi.
int oracle_mla_decode_fp8(int B, int q_len, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                          const uint8_t* kv_fp8, double kv_scale, int64_t num_blocks,
                          int block_size, const int32_t* block_table, int max_blocks,
                          const int32_t* seq_lens, double sm_scale, double* out, double* lse,
                          int n_threads) {
  if (B < 0 || H < 1 || q_len < 1 || kv_fp8 == nullptr || !std::isfinite(kv_scale))
    return ORACLE_ERR_ARG;
  Inputs in{B, q_len * H, q_nope, q_pe, nullptr, num_blocks, block_size,
            block_table, max_blocks, seq_lens, sm_scale, kv_fp8, kv_scale};
  return decode_causal(in, q_len, out, lse, n_threads);
}

// Sparse decode (top-k token selection): request b attends only to the
// tokens listed in topk_indices[b][0..topk), logical positions in its
// sequence shared by all its heads; an entry outside [0, L) is padding and is
// skipped, and an entry listed twice is attended twice. q, out and lse are
// shaped as in oracle_mla_decode. The pages name a sparse MLA backend only;
// the list form, the padding rule and the shared selection are the readings
// taken there.
// With kv_fp8 non-null the cache is the FP8 one of oracle_mla_decode_fp8
// (kv_cache is then ignored).
int oracle_mla_decode_sparse(int B, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                             const uint16_t* kv_cache, int64_t num_blocks, int block_size,
                             const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                             const int32_t* topk_indices, int topk, double sm_scale, double* out,
                             double* lse, int n_threads, const uint8_t* kv_fp8, double kv_scale) {
  if (B < 0 || H < 1 || topk < 0 || (topk > 0 && topk_indices == nullptr)) return ORACLE_ERR_ARG;
  if (kv_fp8 != nullptr && !std::isfinite(kv_scale)) return ORACLE_ERR_ARG;
  Inputs in{B, H, q_nope, q_pe, kv_fp8 != nullptr ? nullptr : kv_cache, num_blocks, block_size,
            block_table, max_blocks, seq_lens, sm_scale, kv_fp8, kv_scale};
  if (!valid_shape(in)) return ORACLE_ERR_ARG;
  set_threads(n_threads);
  const int64_t n = static_cast<int64_t>(B) * H;
  int status = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t r = 0; r < n; ++r) {
    const int b = static_cast<int>(r / H);
    const int h = static_cast<int>(r % H);
    std::vector<int64_t> tokens;
    for (int i = 0; i < topk; ++i) {
      const int64_t t = topk_indices[static_cast<int64_t>(b) * topk + i];
      if (t >= 0 && t < seq_lens[b]) tokens.push_back(t);
    }
    const int rc = attend_tokens(in, b, h, tokens, out + r * kDc, lse + r);
    if (rc != ORACLE_OK) {
#pragma omp critical
      status = rc;
    }
  }
  return status;
}

// E4M3 bytes -> doubles, element by element (NaN for the two NaN codes).
int oracle_e4m3_decode(int64_t n, const uint8_t* bytes, double* out) {
  if (n < 0) return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_to_double(bytes[i]);
  return ORACLE_OK;
}

// Split-KV partial of one (b, h) over tokens [t0, t1): the normalised partial
// output o[512] and that range's log-sum-exp. This is what one split of the
// split-KV decode produces before the reduction step.
int oracle_mla_partial(int B, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                       const uint16_t* kv_cache, int64_t num_blocks, int block_size,
                       const int32_t* block_table, int max_blocks, const int32_t* seq_lens,
                       double sm_scale, int b, int h, int64_t t0, int64_t t1, double* o,
                       double* lse) {
  Inputs in{B, H, q_nope, q_pe, kv_cache, num_blocks, block_size,
            block_table, max_blocks, seq_lens, sm_scale};
  if (!valid_shape(in) || b < 0 || b >= B || h < 0 || h >= H) return ORACLE_ERR_ARG;
  if (t0 < 0 || t1 > seq_lens[b] || t0 > t1) return ORACLE_ERR_ARG;
  return attend_range(in, b, h, t0, t1, o, lse);
}

// Reduction of n split partials (o_parts[n, 512], lse_parts[n]) of one
// (b, h): lse = ln sum_i exp(lse_i); out = sum_i exp(lse_i - lse) * o_i.
// Partials with lse_i = -inf carry no tokens and get weight 0; if all are
// -inf the result is out = 0, lse = -inf.
int oracle_mla_combine(int n, const double* o_parts, const double* lse_parts, double* o,
                       double* lse) {
  if (n < 0) return ORACLE_ERR_ARG;
  for (int j = 0; j < kDc; ++j) o[j] = 0.0;
  double mx = -std::numeric_limits<double>::infinity();
  for (int i = 0; i < n; ++i)
    if (lse_parts[i] > mx) mx = lse_parts[i];
  if (n == 0 || mx == -std::numeric_limits<double>::infinity()) {
    *lse = -std::numeric_limits<double>::infinity();
    return ORACLE_OK;
  }
  double z = 0.0;
  for (int i = 0; i < n; ++i) z += std::exp(lse_parts[i] - mx);
  const double total = mx + std::log(z);
  for (int i = 0; i < n; ++i) {
    if (lse_parts[i] == -std::numeric_limits<double>::infinity()) continue;
    const double w = std::exp(lse_parts[i] - total);
    for (int j = 0; j < kDc; ++j) o[j] += w * o_parts[static_cast<int64_t>(i) * kDc + j];
  }
  *lse = total;
  return ORACLE_OK;
}

// Independent second path for tiny inputs: long double throughout, the K rows
// of each request copied into a dense [L, 576] matrix first, every score
// formed as one dot product of the concatenated query [q_nope | q_pe] with a
// dense row, and exp taken without subtracting the maximum (valid only while
// exp(s) cannot overflow, i.e. for small, N(0,1)-sized inputs).
int oracle_mla_decode_bruteforce(int B, int H, const uint16_t* q_nope, const uint16_t* q_pe,
                                 const uint16_t* kv_cache, int64_t num_blocks, int block_size,
                                 const int32_t* block_table, int max_blocks,
                                 const int32_t* seq_lens, double sm_scale, double* out,
                                 double* lse) {
  if (B < 0 || H < 1 || block_size < 1) return ORACLE_ERR_ARG;
  for (int b = 0; b < B; ++b) {
    const int64_t L = seq_lens[b];
    if (L < 0 || L > static_cast<int64_t>(max_blocks) * block_size) return ORACLE_ERR_ARG;
    std::vector<long double> K(static_cast<size_t>(L) * kD);
    for (int64_t t = 0; t < L; ++t) {
      const int32_t blk = block_table[static_cast<int64_t>(b) * max_blocks + t / block_size];
      if (blk < 0 || blk >= num_blocks) return ORACLE_ERR_BAD_BLOCK;
      const uint16_t* src =
          kv_cache + (static_cast<int64_t>(blk) * block_size + t % block_size) * kD;
      for (int d = 0; d < kD; ++d) K[static_cast<size_t>(t) * kD + d] = bf16_to_double(src[d]);
    }
    for (int h = 0; h < H; ++h) {
      long double q[kD];
      for (int d = 0; d < kDc; ++d)
        q[d] = bf16_to_double(q_nope[(static_cast<int64_t>(b) * H + h) * kDc + d]);
      for (int d = 0; d < kDr; ++d)
        q[kDc + d] = bf16_to_double(q_pe[(static_cast<int64_t>(b) * H + h) * kDr + d]);
      double* o = out + (static_cast<int64_t>(b) * H + h) * kDc;
      if (L == 0) {
        for (int j = 0; j < kDc; ++j) o[j] = 0.0;
        lse[static_cast<int64_t>(b) * H + h] = -std::numeric_limits<double>::infinity();
        continue;
      }
      std::vector<long double> e(static_cast<size_t>(L));
      long double z = 0.0L;
      for (int64_t t = 0; t < L; ++t) {
        long double dot = 0.0L;
        for (int d = 0; d < kD; ++d) dot += q[d] * K[static_cast<size_t>(t) * kD + d];
        e[t] = std::exp(static_cast<long double>(sm_scale) * dot);
        z += e[t];
      }
      for (int j = 0; j < kDc; ++j) {
        long double acc = 0.0L;
        for (int64_t t = 0; t < L; ++t) acc += e[t] * K[static_cast<size_t>(t) * kD + j];
        o[j] = static_cast<double>(acc / z);
      }
      lse[static_cast<int64_t>(b) * H + h] = static_cast<double>(std::log(z));
    }
  }
  return ORACLE_OK;
}

}  // extern "C"
