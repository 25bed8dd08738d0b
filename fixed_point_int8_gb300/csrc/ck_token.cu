// The tokenizer ("The inference core", "The forward pass, in order", phases 0 to 2) and the
// text of generated tokens ("Sampling", last paragraph).  Host code: a prompt is tokenized
// once per run, before any position runs, and is not part of the data-parallel path.
//
// Vocabulary: llama2.c's tokenizer file layout (u32 longest token length, then per token an
// f32 score, an i32 byte length and the bytes), `vocab` tokens.  Strings must be distinct.
#include <cstdint>
#include <cstring>
#include <new>
#include <string>
#include <unordered_map>
#include <vector>

#include "../../include/ck.h"

struct ck_tokenizer {
  std::vector<std::string> text;
  std::vector<float> score;
  std::unordered_map<std::string, uint32_t> id_of;
};

namespace {

// True when s[0..n) is valid UTF-8 (no overlong forms, no surrogates, at most U+10FFFF);
// `lens` receives each character's byte length.
bool split_utf8(const uint8_t* s, size_t n, std::vector<uint32_t>* lens) {
  size_t i = 0;
  while (i < n) {
    const uint8_t b = s[i];
    uint32_t k, cp, min_cp;
    if (b < 0x80) {
      k = 1, cp = b, min_cp = 0;
    } else if (b >= 0xC0 && b < 0xE0) {
      k = 2, cp = b & 0x1Fu, min_cp = 0x80;
    } else if (b >= 0xE0 && b < 0xF0) {
      k = 3, cp = b & 0x0Fu, min_cp = 0x800;
    } else if (b >= 0xF0 && b < 0xF8) {
      k = 4, cp = b & 0x07u, min_cp = 0x10000;
    } else {
      return false;
    }
    if (i + k > n) return false;
    for (uint32_t j = 1; j < k; ++j) {
      if ((s[i + j] >> 6) != 2u) return false;
      cp = (cp << 6) | (s[i + j] & 0x3Fu);
    }
    if (cp < min_cp || cp > 0x10FFFFu || (cp >= 0xD800u && cp < 0xE000u)) return false;
    lens->push_back(k);
    i += k;
  }
  return true;
}

int hex_digit(uint8_t c) {
  if (c >= '0' && c <= '9') return c - '0';
  if (c >= 'A' && c <= 'F') return c - 'A' + 10;
  if (c >= 'a' && c <= 'f') return c - 'a' + 10;
  return -1;
}

}  // namespace

extern "C" {

int ck_tokenizer_load(const void* blob, size_t len, uint32_t vocab, ck_tokenizer** out) {
  if (!blob || !out || vocab == 0) return CK_INVALID_ARGUMENT;
  *out = nullptr;
  const uint8_t* b = static_cast<const uint8_t*>(blob);
  ck_tokenizer* t = new (std::nothrow) ck_tokenizer;
  if (!t) return CK_INVALID_ARGUMENT;
  size_t off = 4;
  t->text.reserve(vocab);
  t->score.reserve(vocab);
  for (uint32_t i = 0; i < vocab; ++i) {
    float sc;
    int32_t n;
    if (len < off + 8) {
      delete t;
      return CK_INVALID_FORMAT;
    }
    memcpy(&sc, b + off, 4);
    memcpy(&n, b + off + 4, 4);
    off += 8;
    if (n < 0 || len - off < (size_t)n) {
      delete t;
      return CK_INVALID_FORMAT;
    }
    std::string s(reinterpret_cast<const char*>(b + off), (size_t)n);
    off += (size_t)n;
    if (!t->id_of.emplace(s, i).second) {  // repeated strings make lookups ambiguous
      delete t;
      return CK_INVALID_FORMAT;
    }
    t->text.push_back(std::move(s));
    t->score.push_back(sc);
  }
  *out = t;
  return CK_OK;
}

void ck_tokenizer_free(ck_tokenizer* t) { delete t; }

int ck_encode(const ck_tokenizer* t, const uint8_t* text, size_t len, uint32_t* ids, uint32_t cap,
              uint32_t* n) {
  if (!t || !n || (len && !text) || (cap && !ids)) return CK_INVALID_ARGUMENT;
  *n = 0;
  if (len > 1024 || (len && memchr(text, 0, len))) return CK_INVALID_PROMPT;
  std::vector<uint32_t> lens;
  if (!split_utf8(text, len, &lens)) return CK_INVALID_PROMPT;
  std::vector<uint32_t> seq;
  seq.push_back(1);  // phase 0: the opening token, then a single space when there is text
  if (len) {
    auto it = t->id_of.find(" ");
    seq.push_back(it != t->id_of.end() ? it->second : (uint32_t)' ' + 3);
  }
  size_t pos = 0;  // phase 1: one token per character, or one per byte
  for (uint32_t k : lens) {
    auto it = t->id_of.find(std::string(reinterpret_cast<const char*>(text + pos), k));
    if (it != t->id_of.end()) {
      seq.push_back(it->second);
    } else {
      for (uint32_t j = 0; j < k; ++j) seq.push_back((uint32_t)text[pos + j] + 3);
    }
    pos += k;
  }
  for (;;) {  // phase 2: the best-scoring pair merges, until none does
    size_t at = SIZE_MAX;
    uint32_t merged = 0;
    float best = 0.f;
    std::string joined;
    for (size_t i = 0; i + 1 < seq.size(); ++i) {
      joined.assign(t->text[seq[i]]);
      joined += t->text[seq[i + 1]];
      auto it = t->id_of.find(joined);
      if (it == t->id_of.end()) continue;
      const float sc = t->score[it->second];
      if (at == SIZE_MAX || sc > best) {  // strictly better: the leftmost of equals stays
        at = i;
        merged = it->second;
        best = sc;
      }
    }
    if (at == SIZE_MAX) break;
    seq[at] = merged;
    seq.erase(seq.begin() + (long)at + 1);
  }
  *n = (uint32_t)seq.size();
  if (seq.size() > cap) return CK_BUFFER_TOO_SMALL;
  memcpy(ids, seq.data(), 4 * seq.size());
  return CK_OK;
}

int ck_decode(const ck_tokenizer* t, uint32_t prev, const uint32_t* ids, uint32_t n, uint8_t* out,
              size_t cap, size_t* n_bytes) {
  if (!t || !n_bytes || (n && !ids) || (cap && !out)) return CK_INVALID_ARGUMENT;
  size_t w = 0;
  for (uint32_t i = 0; i < n; ++i) {
    const uint32_t tok = ids[i];
    const uint32_t before = prev;
    prev = tok;
    if (tok >= t->text.size() || tok == 1 || tok == 2) continue;  // no text
    const std::string& s = t->text[tok];
    size_t from = (before == 1 && !s.empty() && s[0] == ' ') ? 1 : 0;
    uint8_t single;
    const uint8_t* src = reinterpret_cast<const uint8_t*>(s.data()) + from;
    size_t k = s.size() - from;
    if (k == 6 && src[0] == '<' && src[1] == '0' && src[2] == 'x' && src[5] == '>') {
      const int hi = hex_digit(src[3]), lo = hex_digit(src[4]);
      if (hi >= 0 && lo >= 0) {
        single = (uint8_t)(hi * 16 + lo);
        src = &single;
        k = 1;
      }
    }
    for (size_t j = 0; j < k; ++j, ++w)
      if (w < cap) out[w] = src[j];
  }
  *n_bytes = w;
  return w > cap ? CK_BUFFER_TOO_SMALL : CK_OK;
}

}  // extern "C"
