// Conversion between this library's state ("CKSTATE1", ids mode) and the page's state
// ("The resumable state": CURTAST2, a 128-byte header and text-mode buffers), at position
// boundaries, so that a run can move to a target that runs the page's state -- which can
// stop at any phase boundary, mid-layer included -- and come back.  Host code on host
// copies of the states (ck_state_download / ck_state_upload move them).
#include <cstdint>
#include <cstring>
#include <vector>

#include "ck_internal.cuh"

using namespace ck;

namespace {

// The page's header fields (offsets from the start of the state).
constexpr uint32_t kPPhase = 8, kPLayer = 12, kPRow = 16, kPPos = 20, kPToken = 24, kPPromptBytes = 28,
                   kPPromptTokens = 32, kPMaxTok = 36, kPTemp = 40, kPGenerated = 44, kPTextBytes = 48,
                   kPSeed = 72, kPTurns = 80, kPMaxScore = 88, kPChosen = 96, kPSum = 104, kPDraw = 112;

struct PageLayout {
  uint64_t prompt, ptok, out, text, x, logits, k, v, size;
  uint32_t cache;
};

uint64_t up8(uint64_t n) { return (n + 7) & ~7ull; }

// The page's buffers, each at a multiple of eight bytes: prompt u8[bytes], prompt tokens
// u32[bytes + 2], output tokens u32[max tokens], output text u8[128 max tokens], activations
// and three working vectors i64[dim], gate and up i64[hidden], logits i64[vocab], scores
// i64[cache], keys and values i32[layers][cache][kv_dim]; cache = min(bytes + max + 1,
// context).
PageLayout page_layout(const ck_config& c, uint32_t kv_dim, uint32_t prompt_bytes, uint32_t max_tokens) {
  PageLayout L;
  uint64_t cache = (uint64_t)prompt_bytes + max_tokens + 1;
  if (cache > c.context) cache = c.context;
  uint64_t n = 128;
  L.prompt = n; n = up8(n + prompt_bytes);
  L.ptok = n; n = up8(n + 4ull * (prompt_bytes + 2));
  L.out = n; n = up8(n + 4ull * max_tokens);
  L.text = n; n = up8(n + 128ull * max_tokens);
  L.x = n; n = up8(n + 32ull * c.dim);
  n = up8(n + 16ull * c.hidden);
  L.logits = n; n = up8(n + 8ull * c.vocab);
  n = up8(n + 8 * cache);
  L.k = n; n = up8(n + 4ull * c.layers * cache * kv_dim);
  L.v = n; n = up8(n + 4ull * c.layers * cache * kv_dim);
  L.size = n;
  L.cache = (uint32_t)cache;
  return L;
}

template <typename T>
T get(const uint8_t* b, uint64_t off) {
  T v;
  memcpy(&v, b + off, sizeof(T));
  return v;
}
template <typename T>
void put(uint8_t* b, uint64_t off, T v) {
  memcpy(b + off, &v, sizeof(T));
}

bool config_matches(const ck_config& c, const uint8_t* st) {
  for (int i = 0; i < 7; ++i)
    if (get<uint32_t>(st, kHConfig + 4 * i) != (&c.dim)[i]) return false;
  return true;
}

}  // namespace

extern "C" {

int ck_page_size(const ck_model* m, uint32_t prompt_bytes, uint32_t max_tokens, size_t* out) {
  ck_config c;
  if (!m || !out || ck_model_config(m, &c) != CK_OK) return CK_INVALID_ARGUMENT;
  const uint32_t kv_dim = c.dim / c.heads * c.kv_heads;
  *out = page_layout(c, kv_dim, prompt_bytes, max_tokens).size;
  return CK_OK;
}

int ck_state_to_page(const ck_model* m, const ck_tokenizer* t, const void* host_state, size_t len,
                     const uint8_t* prompt, size_t prompt_len, void* host_page, size_t page_len) {
  ck_config c;
  if (!m || !t || !host_state || !host_page || (prompt_len && !prompt) || ck_model_config(m, &c) != CK_OK)
    return CK_INVALID_ARGUMENT;
  const uint8_t* st = static_cast<const uint8_t*>(host_state);
  uint8_t* pg = static_cast<uint8_t*>(host_page);
  if (len < kHeaderBytes || memcmp(st, "CKSTATE1", 8) != 0 || !config_matches(c, st)) return CK_INVALID_STATE;
  const uint32_t np = get<uint32_t>(st, kHNPrompt), mt = get<uint32_t>(st, kHMaxTok);
  const StateLayout lay = state_layout(c, np, mt);
  if (len != lay.size) return CK_INVALID_STATE;
  const uint32_t phase = get<uint32_t>(st, kHPhase);
  if (phase != CK_PHASE_RUNNING && phase != CK_PHASE_DONE) return CK_INVALID_STATE;  // failed
  // the page's runs end at tokens 1 and 2: only states made to do the same convert
  if (!(get<uint32_t>(st, kHFlags) & CK_FLAG_STOP_TOKENS)) return CK_INVALID_STATE;
  // the state's ids must be the prompt's tokens
  std::vector<uint32_t> ids(prompt_len + 2);
  uint32_t n = 0;
  int rc = ck_encode(t, prompt, prompt_len, ids.data(), (uint32_t)ids.size(), &n);
  if (rc) return rc;
  if (n != np || memcmp(ids.data(), st + lay.prompt, 4ull * np) != 0) return CK_INVALID_STATE;
  const uint32_t kv_dim = c.dim / c.heads * c.kv_heads, hd = c.dim / c.heads;
  const PageLayout P = page_layout(c, kv_dim, (uint32_t)prompt_len, mt);
  if (page_len != P.size) return CK_BUFFER_TOO_SMALL;
  if (lay.cache > P.cache) return CK_CONTEXT_EXCEEDED;
  memset(pg, 0, page_len);
  memcpy(pg, "CURTAST2", 8);
  const uint32_t pos = get<uint32_t>(st, kHPosition), gen = get<uint32_t>(st, kHGenerated);
  const uint32_t* outs = reinterpret_cast<const uint32_t*>(st + lay.out);
  put<uint32_t>(pg, kPPhase, phase == CK_PHASE_DONE ? 20u : 3u);
  put<uint32_t>(pg, kPLayer, 0);
  put<uint32_t>(pg, kPRow, 0);
  put<uint32_t>(pg, kPPos, phase == CK_PHASE_DONE ? pos - 1 : pos);
  const uint32_t cur = pos < np ? ids[pos] : (gen ? outs[gen - 1] : 0u);
  put<uint32_t>(pg, kPToken, phase == CK_PHASE_DONE ? (gen ? outs[gen - 1] : 0u) : cur);
  put<uint32_t>(pg, kPPromptBytes, (uint32_t)prompt_len);
  put<uint32_t>(pg, kPPromptTokens, np);
  put<uint32_t>(pg, kPMaxTok, mt);
  put<uint32_t>(pg, kPTemp, get<uint32_t>(st, kHTemp));
  put<uint32_t>(pg, kPGenerated, gen);
  put<uint64_t>(pg, kPSeed, get<uint64_t>(st, kHSeed));
  put<uint64_t>(pg, kPTurns, get<uint64_t>(st, kHTurns));
  put<int64_t>(pg, kPMaxScore, get<int64_t>(st, kHMaxLogit));
  put<uint32_t>(pg, kPChosen, gen ? outs[gen - 1] : 0u);
  put<uint64_t>(pg, kPSum, get<uint64_t>(st, kHExpSum));
  put<uint64_t>(pg, kPDraw, get<uint64_t>(st, kHDraw));
  memcpy(pg + P.prompt, prompt, prompt_len);
  memcpy(pg + P.ptok, ids.data(), 4ull * np);
  memcpy(pg + P.out, outs, 4ull * gen);
  size_t tb = 0;
  rc = ck_decode(t, ids[np - 1], outs, gen, pg + P.text, 128ull * mt, &tb);
  if (rc) return rc;
  put<uint32_t>(pg, kPTextBytes, (uint32_t)tb);
  memcpy(pg + P.x, st + lay.x, 8ull * c.dim);
  memcpy(pg + P.logits, st + lay.logits, 8ull * c.vocab);
  // caches: [layer][kv head][position][element] here, [layer][position][kv_dim] there
  for (int which = 0; which < 2; ++which) {
    const int32_t* src = reinterpret_cast<const int32_t*>(st + (which ? lay.v : lay.k));
    int32_t* dst = reinterpret_cast<int32_t*>(pg + (which ? P.v : P.k));
    for (uint32_t l = 0; l < c.layers; ++l)
      for (uint32_t p = 0; p < lay.cache; ++p)
        for (uint32_t e = 0; e < kv_dim; ++e)
          dst[((size_t)l * P.cache + p) * kv_dim + e] =
              src[(size_t)l * lay.cache * kv_dim + cache_word(e, p, hd, lay.cache)];
  }
  return CK_OK;
}

int ck_state_from_page(const ck_model* m, const void* host_page, size_t page_len, void* host_state, size_t len) {
  ck_config c;
  if (!m || !host_page || !host_state || ck_model_config(m, &c) != CK_OK) return CK_INVALID_ARGUMENT;
  const uint8_t* pg = static_cast<const uint8_t*>(host_page);
  uint8_t* st = static_cast<uint8_t*>(host_state);
  if (page_len < 128 || memcmp(pg, "CURTAST2", 8) != 0) return CK_INVALID_STATE;
  const uint32_t phase = get<uint32_t>(pg, kPPhase);
  // a position boundary: the start of a position, or done
  if ((phase != 3 && phase != 20) || (phase == 3 && get<uint32_t>(pg, kPLayer) != 0)) return CK_INVALID_STATE;
  const uint32_t pb = get<uint32_t>(pg, kPPromptBytes), mt = get<uint32_t>(pg, kPMaxTok);
  const uint32_t np = get<uint32_t>(pg, kPPromptTokens), gen = get<uint32_t>(pg, kPGenerated);
  const uint32_t kv_dim = c.dim / c.heads * c.kv_heads, hd = c.dim / c.heads;
  const PageLayout P = page_layout(c, kv_dim, pb, mt);
  if (page_len != P.size || np == 0 || mt == 0 || (uint64_t)np + mt - 1 > c.context) return CK_INVALID_STATE;
  const StateLayout lay = state_layout(c, np, mt);
  if (len != lay.size) return CK_BUFFER_TOO_SMALL;
  if (lay.cache > P.cache) return CK_INVALID_STATE;
  const uint32_t ppos = get<uint32_t>(pg, kPPos);
  const uint32_t pos = phase == 20 ? ppos + 1 : ppos;  // the next position to run
  if (pos > lay.cache || gen != (pos + 1 > np ? pos + 1 - np : 0u)) return CK_INVALID_STATE;
  memset(st, 0, len);
  memcpy(st, "CKSTATE1", 8);
  put<uint32_t>(st, kHPhase, phase == 20 ? CK_PHASE_DONE : CK_PHASE_RUNNING);
  put<uint32_t>(st, kHPosition, pos);
  put<uint32_t>(st, kHNPrompt, np);
  put<uint32_t>(st, kHMaxTok, mt);
  put<uint32_t>(st, kHCache, lay.cache);
  put<uint32_t>(st, kHGenerated, gen);
  put<uint32_t>(st, kHFlags, CK_FLAG_STOP_TOKENS);  // the page's runs end at tokens 1 and 2
  put<uint32_t>(st, kHTemp, get<uint32_t>(pg, kPTemp));
  const uint32_t* outs = reinterpret_cast<const uint32_t*>(pg + P.out);
  put<uint32_t>(st, kHLastTok, gen ? outs[gen - 1] : 0xFFFFFFFFu);
  put<uint64_t>(st, kHSeed, get<uint64_t>(pg, kPSeed));
  put<uint64_t>(st, kHTurns, get<uint64_t>(pg, kPTurns));
  put<uint64_t>(st, kHErrKey, kNoError);
  put<int64_t>(st, kHMaxLogit, get<int64_t>(pg, kPMaxScore));
  for (int i = 0; i < 7; ++i) put<uint32_t>(st, kHConfig + 4 * i, (&c.dim)[i]);
  put<uint64_t>(st, kHExpSum, get<uint64_t>(pg, kPSum));
  put<uint64_t>(st, kHDraw, get<uint64_t>(pg, kPDraw));
  memcpy(st + lay.prompt, pg + P.ptok, 4ull * np);
  memcpy(st + lay.out, outs, 4ull * gen);
  memcpy(st + lay.x, pg + P.x, 8ull * c.dim);
  memcpy(st + lay.logits, pg + P.logits, 8ull * c.vocab);
  for (int which = 0; which < 2; ++which) {
    const int32_t* src = reinterpret_cast<const int32_t*>(pg + (which ? P.v : P.k));
    int32_t* dst = reinterpret_cast<int32_t*>(st + (which ? lay.v : lay.k));
    for (uint32_t l = 0; l < c.layers; ++l)
      for (uint32_t p = 0; p < lay.cache; ++p)
        for (uint32_t e = 0; e < kv_dim; ++e)
          dst[(size_t)l * lay.cache * kv_dim + cache_word(e, p, hd, lay.cache)] =
              src[((size_t)l * P.cache + p) * kv_dim + e];
  }
  return CK_OK;
}

}  // extern "C"
