// CSA2 step oracle: a plain, slow CPU statement of what the step computes.
//
// TEST INFRASTRUCTURE.  Only the tests, the smoke check and the benchmark's CPU
// baseline load this library.  It shares no code with the CUDA path: no headers,
// tables or helpers are common to both.  Everything is written for clarity, not
// speed: no blocking, no fusion, no reordering beyond what each definition says.
//
// Sources (web pages on DeepSeek-V4.1-Flash; cited by title and section):
//  [AIM]  "DeepSeek AI released DeepSeek-V4.1-Flash with 1M context, FP4" (ai-maestro.online),
//         sections "Causal Encoder-Decoder architecture", "Compressed Sparse Attention 2",
//         "FP4 KV, Bounded Replay, and other extensions".
//  [WPN]  "DeepSeek V4.1 Flash Specs: KV Cache Compression Explained" (wpnews.pro),
//         section "What is Compressed Sparse Attention 2 CSA2?".
//  [KCH]  "DeepSeek V4.1 Flash Deep Dive: The Technical Path to 437x KV Cache Compression"
//         (kongchang.com), section "Compressed Absorption Attention (2nd Gen)".
//  [CTC]  "DeepSeek V4.1 Flash: Reducing KV Cache to 890 Bytes per Token", section
//         "Architectural Breakthroughs in Memory Efficiency" ("4-bit Quantization").
//
// The pages fix the structure (modes, Top-512, 2,048 blocks of 8 tokens, E2M1 codes with
// one E4M3 scale per 16 channels, a 128-token window).  They give no formula for the
// indexer score, no dimensions and no rounding or tie rules; those are the workload's
// definitions, restated where they are used:
//   d = 512 latent channels shared as K and V, 16 main heads, indexer Q of 4 heads x 128
//   bf16 with fp32 head weights, s_t = sum_h w_h * relu(qI_h . KI_t), Top-K ties broken by
//   the lower position, scale = E4M3(amax / 6) with round-to-nearest-even.
// Readings taken where everything is silent are marked READING in the comments.
//
// Build: g++ -O2 -std=c++17 -ffp-contract=off -fPIC -shared -pthread (no fused multiply-add
// is formed implicitly; std::fma is used exactly where the canonical score order says so).

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <numeric>
#include <thread>
#include <vector>

namespace {

constexpr int kD = 512;        // main latent width (K and V share it)
constexpr int kGroup = 16;     // channels per E4M3 scale
constexpr int kCodeBytes = kD / 2;
constexpr int kScaleBytes = kD / kGroup;
constexpr int kHI = 4;         // indexer heads
constexpr int kDI = 128;       // indexer width
constexpr int kH = 16;         // main heads
constexpr int kBlock = 8;      // tokens per block in the hierarchical indexer

enum { MODE_FULL = 0, MODE_REINDEX = 1, MODE_REUSE = 2 };

float bf16_to_f32(uint16_t b) {
  uint32_t u = uint32_t(b) << 16;
  float f;
  std::memcpy(&f, &u, 4);
  return f;
}

// float -> bf16, round to nearest, ties to even (inputs finite).
uint16_t f32_to_bf16(float f) {
  uint32_t u;
  std::memcpy(&u, &f, 4);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return uint16_t(u >> 16);
}

// ---------------------------------------------------------------------------
// FP8 E4M3 (the "FN" variant of the OCP 8-bit formats, as used by NVFP4 block scales):
// sign, 4 exponent bits with bias 7, 3 mantissa bits, no infinities, S.1111.111 = NaN,
// largest finite 448.  [AIM] "FP4 KV...": one E4M3 scale per 16 channels.
// ---------------------------------------------------------------------------
double e4m3_value(uint8_t b) {
  const int s = b >> 7, e = (b >> 3) & 15, m = b & 7;
  if (e == 15 && m == 7) return std::nan("");
  double v = (e == 0) ? std::ldexp(double(m), -9)               // subnormal: m/8 * 2^-6
                      : std::ldexp(1.0 + m / 8.0, e - 7);
  return s ? -v : v;
}

// Round a finite value to E4M3 with round-to-nearest-even, saturating to +-448.
uint8_t e4m3_encode(float v) {
  const uint8_t sign = std::signbit(v) ? 0x80 : 0x00;
  const double a = std::fabs(double(v));
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);                        // a = f * 2^e2, f in [0.5, 1)
  const int E = std::max(e2 - 1, -6);        // binade exponent, clamped at the normal minimum
  const double quantum = std::ldexp(1.0, E - 3);
  double r = std::nearbyint(a / quantum) * quantum;   // a/quantum is exact; RNE by default mode
  if (r > 448.0) r = 448.0;
  if (r == 0.0) return sign;
  uint8_t mag;
  if (r < std::ldexp(1.0, -6)) {
    mag = uint8_t(r / std::ldexp(1.0, -9));  // subnormal: r = m * 2^-9
  } else {
    int f2;
    std::frexp(r, &f2);
    const int Er = f2 - 1;
    const int m = int(r / std::ldexp(1.0, Er) * 8.0) - 8;
    mag = uint8_t(((Er + 7) << 3) | m);
  }
  return uint8_t(sign | mag);
}

// ---------------------------------------------------------------------------
// FP4 E2M1: sign, 2 exponent bits with bias 1, 1 mantissa bit.  Magnitudes
// {0, 0.5, 1, 1.5, 2, 3, 4, 6}.  [AIM] "FP4 KV...": "quantises to E2M1".
// ---------------------------------------------------------------------------
const float kE2M1[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};

float e2m1_value(uint8_t nib) {
  const float v = kE2M1[nib & 7];
  return (nib & 8) ? -v : v;
}

// Round to E2M1 with round-to-nearest-even, saturating to +-6.  The sign bit follows the
// input's sign, also when the magnitude rounds to zero (READING).
uint8_t e2m1_encode(float v) {
  const uint8_t sign = std::signbit(v) ? 8 : 0;
  const double a = std::fabs(double(v));
  if (a == 0.0) return sign;
  int e2;
  std::frexp(a, &e2);
  const int E = std::max(e2 - 1, 0);         // binade exponent; [0, 1) shares quantum 0.5
  const double quantum = std::ldexp(1.0, E - 1);
  double r = std::nearbyint(a / quantum) * quantum;
  if (r > 6.0) r = 6.0;
  for (uint8_t k = 0; k < 8; ++k)
    if (double(kE2M1[k]) == r) return uint8_t(sign | k);
  return sign;  // unreachable for finite input
}

// ---------------------------------------------------------------------------
// NVFP4-without-global-scale quantisation of one 512-channel row ([AIM] "FP4 KV...",
// [WPN] "What is CSA2?": "one E4M3 scaling factor applied per 16 channels").
// Per 16-channel group: amax = max |x|; s8 = E4M3_RNE_satfinite(amax / 6) with the
// quotient formed in fp32; s = value(s8); code_i = E2M1_RNE_satfinite(x_i / s) with the
// quotient formed in fp32 (READING: divide by the decoded scale, so that dequantisation
// x_hat = E2M1(code) * s inverts it).  A group whose scale rounds to zero gets all-zero
// codes.  Codes are packed two per byte, the even channel in the low nibble (READING).
// ---------------------------------------------------------------------------
void quantize_row(const uint16_t* x, uint8_t* codes, uint8_t* scales) {
  for (int g = 0; g < kScaleBytes; ++g) {
    float amax = 0.0f;
    for (int i = 0; i < kGroup; ++i) amax = std::max(amax, std::fabs(bf16_to_f32(x[g * kGroup + i])));
    const float s32 = amax / 6.0f;
    const uint8_t sb = e4m3_encode(s32);
    const float s = float(e4m3_value(sb));
    scales[g] = sb;
    uint8_t nib[kGroup];
    for (int i = 0; i < kGroup; ++i) {
      const float xi = bf16_to_f32(x[g * kGroup + i]);
      nib[i] = (s == 0.0f) ? 0 : e2m1_encode(xi / s);
    }
    for (int i = 0; i < kGroup; i += 2)
      codes[(g * kGroup + i) / 2] = uint8_t(nib[i] | (nib[i + 1] << 4));
  }
}

// Dequantised value of channel c of a stored row, as a double (exact; also exact in bf16).
double dequant_channel(const uint8_t* codes, const uint8_t* scales, int c) {
  const uint8_t byte = codes[c / 2];
  const uint8_t nib = (c & 1) ? (byte >> 4) : (byte & 15);
  return double(e2m1_value(nib)) * e4m3_value(scales[c / kGroup]);
}

// ---------------------------------------------------------------------------
// Indexer score s_t = sum_h w_h * relu(qI_h . KI_t), the workload's definition of the
// lightning-indexer score of indexer Q against cached indexer K ([AIM] "Compressed Sparse
// Attention 2": Full layers select with indexer K, Reindex layers rescore with their own
// indexer Q).  READING (canonical fp32 order; the pages give no order):
//   per head, eight partial sums p_j, each a chain of fused multiply-adds over channels
//   16j .. 16j+15 in increasing order starting from +0;  dot = ((p0+p1)+(p2+p3)) +
//   ((p4+p5)+(p6+p7));  r_h = dot > 0 ? dot : +0;  s = (w0*r0 + w1*r1) + (w2*r2 + w3*r3)
//   with every product and sum rounded to fp32.
// ---------------------------------------------------------------------------
float score_one(const uint16_t* qI, const float* w, const uint16_t* k) {
  float r[kHI];
  for (int h = 0; h < kHI; ++h) {
    float p[8];
    for (int j = 0; j < 8; ++j) {
      float acc = 0.0f;
      for (int c = 16 * j; c < 16 * j + 16; ++c)
        acc = std::fma(bf16_to_f32(qI[h * kDI + c]), bf16_to_f32(k[c]), acc);
      p[j] = acc;
    }
    const float dot = ((p[0] + p[1]) + (p[2] + p[3])) + ((p[4] + p[5]) + (p[6] + p[7]));
    r[h] = dot > 0.0f ? dot : 0.0f;
  }
  const float m0 = w[0] * r[0], m1 = w[1] * r[1], m2 = w[2] * r[2], m3 = w[3] * r[3];
  return (m0 + m1) + (m2 + m3);
}

// ---------------------------------------------------------------------------
// Exact Top-K ([AIM] "Compressed Sparse Attention 2": "selects fresh Top-512 indices").
// Order: larger score first, equal scores by lower position (the workload's tie rule;
// -0 and +0 compare equal).  The result is the first min(K, n) entries, returned in
// ascending position order (READING), padded with -1.
// ---------------------------------------------------------------------------
int topk(const float* scores, int64_t n, int k, const int32_t* map, int32_t* out) {
  std::vector<int64_t> order(static_cast<size_t>(n));
  std::iota(order.begin(), order.end(), int64_t(0));
  std::sort(order.begin(), order.end(), [&](int64_t a, int64_t b) {
    if (scores[a] != scores[b]) return scores[a] > scores[b];
    return a < b;
  });
  const int64_t m = std::min<int64_t>(k, n);
  std::vector<int64_t> sel(order.begin(), order.begin() + m);
  std::sort(sel.begin(), sel.end());
  for (int i = 0; i < k; ++i)
    out[i] = (i < m) ? int32_t(map ? map[sel[size_t(i)]] : sel[size_t(i)]) : -1;
  return int(m);
}

// ---------------------------------------------------------------------------
// Hierarchical Sparse Indexer ([AIM] "Compressed Sparse Attention 2": the Full layer builds
// a candidate pool of up to 16,384 positions, 2,048 blocks of eight tokens; later Reindex
// layers score the bounded set; [KCH] "Compressed Absorption Attention (2nd Gen)").
// Block key (workload definition): the mean of the block's 8 indexer keys; READING: summed
// in token order in fp32, multiplied by 0.125 and rounded to bf16.  Only complete blocks
// exist (READING: a partial trailing block is not scored; the window covers it).
// ---------------------------------------------------------------------------
void block_keys(const uint16_t* KI, int64_t T, uint16_t* out) {
  const int64_t nb = T / kBlock;
  for (int64_t b = 0; b < nb; ++b)
    for (int c = 0; c < kDI; ++c) {
      float acc = 0.0f;
      for (int i = 0; i < kBlock; ++i) acc = acc + bf16_to_f32(KI[(b * kBlock + i) * kDI + c]);
      out[b * kDI + c] = f32_to_bf16(acc * 0.125f);
    }
}

// Score the first n_blocks block keys, keep the top min(keep, n_blocks) blocks (ties to the
// lower block) and expand them into ascending token positions.  Returns the pool length.
int block_pool(const uint16_t* qI, const float* w, const uint16_t* bkeys, int64_t n_blocks,
               int keep, int32_t* pool) {
  std::vector<float> s(size_t(std::max<int64_t>(n_blocks, 1)));
  for (int64_t b = 0; b < n_blocks; ++b) s[size_t(b)] = score_one(qI, w, bkeys + b * kDI);
  std::vector<int32_t> blk(static_cast<size_t>(keep));
  const int m = topk(s.data(), n_blocks, keep, nullptr, blk.data());
  for (int i = 0; i < m; ++i)
    for (int r = 0; r < kBlock; ++r) pool[i * kBlock + r] = blk[size_t(i)] * kBlock + r;
  return m * kBlock;
}

// ---------------------------------------------------------------------------
// Attention of one query's 16 heads over the selected FP4 rows plus the sliding-window rows
// ([AIM] "Causal Encoder-Decoder architecture": a 128-token window in every layer;
// "Compressed Sparse Attention 2": every layer keeps its own main Q and window cache).
// Plain definition in fp64: logits l_j = scale * q_h . v_j over the union of the rows
// (READING: no de-duplication; a token may appear both as a selected row and as a window
// row, and K = V = the row), softmax, o_h = sum_j p_j v_j.  With no rows at all the output is
// zero and lse is -inf.
// ---------------------------------------------------------------------------
void attend(const uint16_t* q, const std::vector<std::vector<double>>& rows, float scale,
            double* out, double* lse) {
  const size_t n = rows.size();
  for (int h = 0; h < kH; ++h) {
    if (n == 0) {
      for (int c = 0; c < kD; ++c) out[h * kD + c] = 0.0;
      if (lse) lse[h] = -INFINITY;
      continue;
    }
    std::vector<double> l(n);
    for (size_t j = 0; j < n; ++j) {
      double acc = 0.0;
      for (int c = 0; c < kD; ++c) acc += double(bf16_to_f32(q[h * kD + c])) * rows[j][size_t(c)];
      l[j] = double(scale) * acc;
    }
    const double m = *std::max_element(l.begin(), l.end());
    double den = 0.0;
    for (size_t j = 0; j < n; ++j) { l[j] = std::exp(l[j] - m); den += l[j]; }
    for (int c = 0; c < kD; ++c) {
      double acc = 0.0;
      for (size_t j = 0; j < n; ++j) acc += l[j] * rows[j][size_t(c)];
      out[h * kD + c] = acc / den;
    }
    if (lse) lse[h] = m + std::log(den);
  }
}

std::vector<double> fp4_row(const uint8_t* codes, const uint8_t* scales, int64_t pos) {
  std::vector<double> v(kD);
  for (int c = 0; c < kD; ++c)
    v[size_t(c)] = dequant_channel(codes + pos * kCodeBytes, scales + pos * kScaleBytes, c);
  return v;
}

std::vector<double> bf16_row(const uint16_t* r) {
  std::vector<double> v(kD);
  for (int c = 0; c < kD; ++c) v[size_t(c)] = double(bf16_to_f32(r[c]));
  return v;
}

// A window row kept in 8 bits ([KCH] "Compressed Absorption Attention (2nd Gen)": the sliding
// window is retained in 8-bit precision): every channel one E4M3 value, no scale (READING).
std::vector<double> fp8_row(const uint8_t* r) {
  std::vector<double> v(kD);
  for (int c = 0; c < kD; ++c) v[size_t(c)] = e4m3_value(r[c]);
  return v;
}

// Entries visible to a query at absolute token position p when each cache entry merges
// `ratio` tokens: entry j covers tokens ratio*j .. ratio*j+ratio-1 and is visible iff its last
// token is <= p (READING, causal mask over compressed positions).
int64_t visible_entries(int64_t T, int64_t p, int ratio) {
  return std::max<int64_t>(0, std::min<int64_t>(T, (p + 1) / ratio));
}

// Runs f(0) .. f(n-1) on up to `threads` host threads (interleaved); the order of the calls does
// not matter to any caller (each index writes only its own outputs).
template <typename F>
void parallel_for(int64_t n, int threads, F f) {
  const int nt = int(std::max<int64_t>(1, std::min<int64_t>(threads, n)));
  if (nt == 1) {
    for (int64_t i = 0; i < n; ++i) f(i);
    return;
  }
  std::vector<std::thread> pool_t;
  for (int t = 0; t < nt; ++t)
    pool_t.emplace_back([&, t] { for (int64_t i = t; i < n; i += nt) f(i); });
  for (auto& th : pool_t) th.join();
}

}  // namespace

extern "C" {

double oracle_e4m3_value(uint8_t b) { return e4m3_value(b); }
uint8_t oracle_e4m3_encode(float v) { return e4m3_encode(v); }
float oracle_e2m1_value(uint8_t n) { return e2m1_value(n); }
uint8_t oracle_e2m1_encode(float v) { return e2m1_encode(v); }

void oracle_fp4_quantize(const uint16_t* x, int64_t rows, uint8_t* codes, uint8_t* scales, int threads) {
  // rows are independent: chunks of 1024 rows on the host threads
  const int64_t chunks = (rows + 1023) / 1024;
  parallel_for(chunks, threads, [&](int64_t ch) {
    for (int64_t r = ch * 1024; r < std::min(rows, ch * 1024 + 1024); ++r)
      quantize_row(x + r * kD, codes + r * kCodeBytes, scales + r * kScaleBytes);
  });
}

// 8-bit window rows: each bf16 element to E4M3 (RNE, saturating to +-448), and back (exact).
void oracle_fp8_quantize(const uint16_t* x, int64_t n, uint8_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = e4m3_encode(bf16_to_f32(x[i]));
}
void oracle_fp8_dequantize(const uint8_t* in, int64_t n, uint16_t* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = f32_to_bf16(float(e4m3_value(in[i])));
}

void oracle_fp4_dequantize(const uint8_t* codes, const uint8_t* scales, int64_t rows, uint16_t* out) {
  for (int64_t r = 0; r < rows; ++r)
    for (int c = 0; c < kD; ++c)
      out[r * kD + c] = f32_to_bf16(float(dequant_channel(codes + r * kCodeBytes, scales + r * kScaleBytes, c)));
}

// Scores of one indexer query against n keys: key i is KI row pos[i] (or row i if pos is NULL).
void oracle_index_score(const uint16_t* qI, const float* w, const uint16_t* KI, const int32_t* pos,
                        int64_t n, float* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = score_one(qI, w, KI + int64_t(pos ? pos[i] : i) * kDI);
}

int oracle_topk(const float* scores, int64_t n, int k, const int32_t* map, int32_t* out) {
  return topk(scores, n, k, map, out);
}

// Flat selection of a Full layer for every query row of a batch: the scores of the row's visible
// entries (score_one), then their exact Top-k (topk), exactly as a flat Full layer of
// oracle_group_step selects.  KI [B][cap][128]; qI [B*Nq][4][128]; w [B*Nq][4]; query i of
// sequence b sits at q_pos[b*Nq+i] (or ratio*T_b - Nq + i when q_pos is NULL).  idx [B*Nq][k],
// n_sel [B*Nq] (nullable).  Rows run on up to `threads` host threads.
void oracle_index_select(int B, int Nq, const int64_t* T, int64_t cap, const uint16_t* KI, const uint16_t* qI,
                         const float* w, int ratio, const int32_t* q_pos, int k, int32_t* idx, int32_t* n_sel,
                         int threads) {
  parallel_for(int64_t(B) * Nq, threads, [&](int64_t row) {
    const int64_t b = row / Nq, i = row - b * Nq;
    const int64_t p = q_pos ? q_pos[row] : int64_t(ratio) * T[b] - Nq + i;
    const int64_t nvis = visible_entries(T[b], p, ratio);
    std::vector<float> s(size_t(std::max<int64_t>(nvis, 1)));
    for (int64_t t = 0; t < nvis; ++t) s[size_t(t)] = score_one(qI + row * kHI * kDI, w + row * kHI, KI + (b * cap + t) * kDI);
    const int m = topk(s.data(), nvis, k, nullptr, idx + row * k);
    if (n_sel) n_sel[row] = m;
  });
}

void oracle_block_keys(const uint16_t* KI, int64_t T, uint16_t* out) { block_keys(KI, T, out); }

int oracle_block_pool(const uint16_t* qI, const float* w, const uint16_t* bkeys, int64_t n_blocks,
                      int keep, int32_t* pool) {
  return block_pool(qI, w, bkeys, n_blocks, keep, pool);
}

// Attention of one query over FP4 cache rows idx[0..k) (entries < 0 are skipped) of a
// sequence's cache (codes/scales point at its row 0) plus n_swa bf16 window rows.
void oracle_sparse_attn(const uint16_t* q, const uint8_t* codes, const uint8_t* scales,
                        const int32_t* idx, int k, const uint16_t* swa_rows, int n_swa,
                        float softmax_scale, double* out, double* lse) {
  std::vector<std::vector<double>> rows;
  for (int i = 0; i < k; ++i)
    if (idx[i] >= 0) rows.push_back(fp4_row(codes, scales, idx[i]));
  for (int r = 0; r < n_swa; ++r) rows.push_back(bf16_row(swa_rows + int64_t(r) * kD));
  attend(q, rows, softmax_scale, out, lse);
}

// One CSA2 layer group over a batch ([AIM] "Compressed Sparse Attention 2"; [WPN] "What is
// CSA2?"; [KCH] "Compressed Absorption Attention (2nd Gen)"):
//   Full    - selects fresh Top-K with its own indexer Q over all visible entries, or, when
//             `hierarchical`, first keeps the top `keep` blocks of 8 and selects within the
//             resulting pool (which later Reindex layers reuse);
//   Reindex - rescored with its own indexer Q over the same candidates (the pool, or all
//             visible entries), fresh Top-K;
//   Reuse   - the latest indices, no scoring.
// Every layer attends with its own main Q and its own window rows over the shared FP4 cache.
// Layout (contiguous): codes [B][cap][256], scales [B][cap][32], KI [B][cap][128];
// per-layer tensors are layer-major: q [L][B][Nq][16][512], qI [L][B][Nq][4][128],
// w [L][B][Nq][4], swa [L][B][W-1+Nq][512] (bf16, or E4M3 bytes when swa_fp8); outputs
// out [L][B][Nq][16][512] (fp64),
// lse [L][B][Nq][16] (nullable), idx [L][B][Nq][K], pool [B][Nq][keep*8] and pool_len [B][Nq]
// (nullable unless hierarchical).  Query i of sequence b sits at token position
// q_pos[b*Nq+i], or ratio*T_b - Nq + i when q_pos is NULL.  Window rows of query i are rows
// i .. i+W-1 of its layer's window buffer, of which the last swa_len[b] rows are valid.
// Returns 0, or -1 on bad arguments.
int oracle_group_step(int B, int L, const int32_t* modes, int Nq, int K, int W, int ratio,
                      int hierarchical, int keep, const int64_t* T, int64_t cap,
                      const uint8_t* codes, const uint8_t* scales, const uint16_t* KI,
                      const int32_t* q_pos, const uint16_t* q, const uint16_t* qI, const float* w,
                      const void* swa, const int32_t* swa_len, float softmax_scale,
                      double* out, double* lse, int32_t* idx, int32_t* pool, int32_t* pool_len,
                      int threads, int swa_fp8) {
  if (B <= 0 || L <= 0 || Nq <= 0 || K <= 0 || W < 0 || ratio <= 0) return -1;
  if (modes[0] == MODE_REUSE) return -1;
  if (hierarchical && (modes[0] != MODE_FULL || keep <= 0 || !pool || !pool_len)) return -1;
  const int SW = W - 1 + Nq;
  const int64_t pool_cap = int64_t(keep) * kBlock;

  // Block keys of every sequence first (hierarchical), then every query row on its own: a row's
  // layers depend only on its sequence's cache and block keys, so rows may run in any order.
  std::vector<std::vector<uint16_t>> bk(static_cast<size_t>(B));
  if (hierarchical)
    parallel_for(B, threads, [&](int64_t b) {
      const int64_t Tb = T[b];
      bk[size_t(b)].resize(size_t(std::max<int64_t>(Tb / kBlock, 1)) * kDI);
      block_keys(KI + b * cap * kDI, Tb, bk[size_t(b)].data());
    });

  auto run_row = [&](int64_t row) {
    const int64_t b = row / Nq, i = row - b * Nq;
    const int64_t Tb = T[b];
    const uint8_t* cb = codes + b * cap * kCodeBytes;
    const uint8_t* sb = scales + b * cap * kScaleBytes;
    const uint16_t* kb = KI + b * cap * kDI;
    const int64_t p = q_pos ? q_pos[row] : int64_t(ratio) * Tb - Nq + i;
    const int64_t nvis = visible_entries(Tb, p, ratio);
    int32_t* prow = hierarchical ? pool + row * pool_cap : nullptr;
    int64_t plen = 0;
    int latest = -1;  // layer whose indices are the latest
    for (int l = 0; l < L; ++l) {
      const int64_t lr = int64_t(l) * B * Nq + row;
      int32_t* il = idx + lr * K;
      const int mode = modes[l];
      if (mode == MODE_FULL || mode == MODE_REINDEX) {
        const uint16_t* qil = qI + lr * kHI * kDI;
        const float* wl = w + lr * kHI;
        if (hierarchical) {
          if (mode == MODE_FULL) {
            plen = block_pool(qil, wl, bk[size_t(b)].data(), nvis / kBlock, keep, prow);
            pool_len[row] = int32_t(plen);
          }
          std::vector<float> s(size_t(std::max<int64_t>(plen, 1)));
          for (int64_t t = 0; t < plen; ++t) s[size_t(t)] = score_one(qil, wl, kb + int64_t(prow[t]) * kDI);
          topk(s.data(), plen, K, prow, il);
        } else {
          std::vector<float> s(size_t(std::max<int64_t>(nvis, 1)));
          for (int64_t t = 0; t < nvis; ++t) s[size_t(t)] = score_one(qil, wl, kb + t * kDI);
          topk(s.data(), nvis, K, nullptr, il);
        }
        latest = l;
      } else {
        std::memcpy(il, idx + (int64_t(latest) * B * Nq + row) * K, sizeof(int32_t) * size_t(K));
      }
      // attention rows: selected FP4 entries, then the query's window rows
      std::vector<std::vector<double>> rows;
      for (int j = 0; j < K; ++j)
        if (il[j] >= 0) rows.push_back(fp4_row(cb, sb, il[j]));
      const int64_t wrow0 = (int64_t(l) * B + b) * SW;
      for (int64_t r = i; r < i + W; ++r) {
        if (r < SW - swa_len[b]) continue;
        if (swa_fp8) rows.push_back(fp8_row(static_cast<const uint8_t*>(swa) + (wrow0 + r) * kD));
        else rows.push_back(bf16_row(static_cast<const uint16_t*>(swa) + (wrow0 + r) * kD));
      }
      attend(q + lr * kH * kD, rows, softmax_scale, out + lr * kH * kD, lse ? lse + lr * kH : nullptr);
    }
  };
  parallel_for(int64_t(B) * Nq, threads, run_row);
  return 0;
}

}  // extern "C"
