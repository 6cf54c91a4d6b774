// Composition manifests: a strict JSON reader for the manifest document and
// its validation into an ordered adapter list.  Host code only.
//
// Source: "We propose a content-addressed overlay system" report,
// §"Composition Identity and Manifest Schema" (base model hash, quantization
// profile, runtime tag, ordered adapters with name, file hash, load order and
// merge weight) and §"Failure Modes" (schema errors, version skew and
// duplicates are rejected); "Deep Technical Design" §11 (AdapterManifestV0:
// adapter type LowRank / Sparse, rank, required base checksum).
//
// The document (one JSON object; every key is listed here, any other key is
// rejected, fail-fast as the pages ask for unknown formats):
//   "base_model_hash": "sha256:<64 lowercase hex>"           required
//   "quantization":    "q8_0" | "q4_0" | "q4_K"              required
//   "runtime":         {"name": "ovl-gb300", "version": "v1"} optional, checked
//   "mode":            "stack" | "table"                      optional, "stack"
//   "tokenizer_id", "timestamp_utc": strings                  optional, not used
//   "adapters": [ {                                           required (may be [])
//       "name": string (1..63 bytes, unique)                  required
//       "file_hash": "sha256:<hex>" (unique)                  required
//       "load_order": integer 1..2^31-1 (unique)              required
//       "merge_weight": number (finite as binary32)           required
//       "type": "lora" | "sparse"                             optional, "lora"
//       "rank": integer 1..OVL_MAX_RANK                       optional, checked
//       "required_base_hash": "sha256:<hex>"                  optional, checked
//       "targets": [tensor index, ...]                        optional, checked
//   } ]
// Adapters are applied in increasing load_order.
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <memory>
#include <string>
#include <utility>
#include <vector>

#include "ovl_internal.h"

namespace ovl {
namespace {

constexpr size_t kMaxManifestBytes = 1u << 20;
constexpr int kMaxDepth = 16;

struct JVal {
  enum Kind { kNull, kBool, kNum, kStr, kArr, kObj } kind = kNull;
  bool b = false;
  std::string s;                                   // string value, or the number's lexeme
  std::vector<JVal> arr;
  std::vector<std::pair<std::string, JVal>> obj;
  const JVal* get(const char* k) const {
    for (const auto& kv : obj)
      if (kv.first == k) return &kv.second;
    return nullptr;
  }
};

// Strict JSON (RFC 8259): no comments, no trailing commas, no NaN/Infinity,
// no duplicate keys, nothing after the value but whitespace.
class Reader {
 public:
  Reader(const char* p, size_t n) : p_(p), e_(p + n) {}
  bool parse(JVal* out, std::string* err) {
    if (!value(out, 0)) {
      *err = "manifest is not valid JSON: " + err_;
      return false;
    }
    ws();
    if (p_ != e_) {
      *err = "manifest is not valid JSON: text after the document";
      return false;
    }
    return true;
  }

 private:
  const char* p_;
  const char* e_;
  std::string err_;

  bool fail(const char* m) {
    err_ = m;
    return false;
  }
  void ws() {
    while (p_ < e_ && (*p_ == ' ' || *p_ == '\t' || *p_ == '\n' || *p_ == '\r')) ++p_;
  }
  bool lit(const char* w) {
    const size_t n = std::strlen(w);
    if (static_cast<size_t>(e_ - p_) < n || std::memcmp(p_, w, n) != 0) return false;
    p_ += n;
    return true;
  }
  static int hexv(char c) {
    if (c >= '0' && c <= '9') return c - '0';
    if (c >= 'a' && c <= 'f') return c - 'a' + 10;
    if (c >= 'A' && c <= 'F') return c - 'A' + 10;
    return -1;
  }
  bool str(std::string* out) {
    if (p_ >= e_ || *p_ != '"') return fail("expected a string");
    ++p_;
    out->clear();
    while (true) {
      if (p_ >= e_) return fail("unterminated string");
      const unsigned char c = static_cast<unsigned char>(*p_++);
      if (c == '"') return true;
      if (c < 0x20) return fail("control character in a string");
      if (c != '\\') {
        out->push_back(static_cast<char>(c));
        continue;
      }
      if (p_ >= e_) return fail("unterminated escape");
      const char x = *p_++;
      switch (x) {
        case '"': out->push_back('"'); break;
        case '\\': out->push_back('\\'); break;
        case '/': out->push_back('/'); break;
        case 'b': out->push_back('\b'); break;
        case 'f': out->push_back('\f'); break;
        case 'n': out->push_back('\n'); break;
        case 'r': out->push_back('\r'); break;
        case 't': out->push_back('\t'); break;
        case 'u': {
          if (e_ - p_ < 4) return fail("short \\u escape");
          uint32_t cp = 0;
          for (int i = 0; i < 4; ++i) {
            const int h = hexv(p_[i]);
            if (h < 0) return fail("bad \\u escape");
            cp = cp * 16 + static_cast<uint32_t>(h);
          }
          p_ += 4;
          if (cp >= 0xD800 && cp <= 0xDFFF) return fail("surrogate \\u escapes are not accepted");
          if (cp < 0x80) {
            out->push_back(static_cast<char>(cp));
          } else if (cp < 0x800) {
            out->push_back(static_cast<char>(0xC0 | (cp >> 6)));
            out->push_back(static_cast<char>(0x80 | (cp & 63)));
          } else {
            out->push_back(static_cast<char>(0xE0 | (cp >> 12)));
            out->push_back(static_cast<char>(0x80 | ((cp >> 6) & 63)));
            out->push_back(static_cast<char>(0x80 | (cp & 63)));
          }
          break;
        }
        default: return fail("unknown escape");
      }
    }
  }
  bool num(std::string* out) {
    const char* s = p_;
    if (p_ < e_ && *p_ == '-') ++p_;
    if (p_ >= e_) return fail("bad number");
    if (*p_ == '0') {
      ++p_;
    } else if (*p_ >= '1' && *p_ <= '9') {
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    } else {
      return fail("bad number");
    }
    if (p_ < e_ && *p_ == '.') {
      ++p_;
      if (p_ >= e_ || *p_ < '0' || *p_ > '9') return fail("bad number");
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    }
    if (p_ < e_ && (*p_ == 'e' || *p_ == 'E')) {
      ++p_;
      if (p_ < e_ && (*p_ == '+' || *p_ == '-')) ++p_;
      if (p_ >= e_ || *p_ < '0' || *p_ > '9') return fail("bad number");
      while (p_ < e_ && *p_ >= '0' && *p_ <= '9') ++p_;
    }
    out->assign(s, p_);
    return true;
  }
  bool value(JVal* v, int depth) {
    if (depth > kMaxDepth) return fail("nesting too deep");
    ws();
    if (p_ >= e_) return fail("unexpected end");
    const char c = *p_;
    if (c == '{') {
      ++p_;
      v->kind = JVal::kObj;
      ws();
      if (p_ < e_ && *p_ == '}') {
        ++p_;
        return true;
      }
      while (true) {
        ws();
        std::string k;
        if (!str(&k)) return false;
        for (const auto& kv : v->obj)
          if (kv.first == k) return fail("duplicate key");
        ws();
        if (p_ >= e_ || *p_ != ':') return fail("expected ':'");
        ++p_;
        JVal item;
        if (!value(&item, depth + 1)) return false;
        v->obj.emplace_back(std::move(k), std::move(item));
        ws();
        if (p_ < e_ && *p_ == ',') {
          ++p_;
          continue;
        }
        if (p_ < e_ && *p_ == '}') {
          ++p_;
          return true;
        }
        return fail("expected ',' or '}'");
      }
    }
    if (c == '[') {
      ++p_;
      v->kind = JVal::kArr;
      ws();
      if (p_ < e_ && *p_ == ']') {
        ++p_;
        return true;
      }
      while (true) {
        JVal item;
        if (!value(&item, depth + 1)) return false;
        v->arr.push_back(std::move(item));
        ws();
        if (p_ < e_ && *p_ == ',') {
          ++p_;
          continue;
        }
        if (p_ < e_ && *p_ == ']') {
          ++p_;
          return true;
        }
        return fail("expected ',' or ']'");
      }
    }
    if (c == '"') {
      v->kind = JVal::kStr;
      return str(&v->s);
    }
    if (lit("true")) {
      v->kind = JVal::kBool;
      v->b = true;
      return true;
    }
    if (lit("false")) {
      v->kind = JVal::kBool;
      return true;
    }
    if (lit("null")) {
      v->kind = JVal::kNull;
      return true;
    }
    v->kind = JVal::kNum;
    return num(&v->s);
  }
};

ovl_status bad(std::string* err, ovl_status code, const std::string& m) {
  *err = m;
  return code;
}

// "sha256:" followed by 64 lowercase hex digits.
bool parse_hash(const JVal* v, uint8_t out[32]) {
  if (!v || v->kind != JVal::kStr || v->s.size() != 7 + 64 || v->s.compare(0, 7, "sha256:") != 0) return false;
  for (int i = 0; i < 32; ++i) {
    int hv[2];
    for (int k = 0; k < 2; ++k) {
      const char c = v->s[7 + 2 * i + k];
      if (c >= '0' && c <= '9') hv[k] = c - '0';
      else if (c >= 'a' && c <= 'f') hv[k] = c - 'a' + 10;
      else return false;
    }
    out[i] = static_cast<uint8_t>(hv[0] * 16 + hv[1]);
  }
  return true;
}

// A JSON integer (no fraction, no exponent) in [lo, hi].
bool parse_int(const JVal* v, int64_t lo, int64_t hi, int64_t* out) {
  if (!v || v->kind != JVal::kNum || v->s.find_first_of(".eE") != std::string::npos || v->s.size() > 18) return false;
  const long long x = std::strtoll(v->s.c_str(), nullptr, 10);
  if (x < lo || x > hi) return false;
  *out = x;
  return true;
}

bool only_keys(const JVal& o, std::initializer_list<const char*> keys, std::string* which) {
  for (const auto& kv : o.obj) {
    bool known = false;
    for (const char* k : keys) known = known || kv.first == k;
    if (!known) {
      *which = kv.first;
      return false;
    }
  }
  return true;
}

}  // namespace

ovl_status parse_manifest(const char* text, size_t len, Manifest* out, std::string* err) {
  if (!text || !out) return bad(err, OVL_E_ARG, "null manifest");
  if (len > kMaxManifestBytes) return bad(err, OVL_E_ARG, "manifest larger than 1 MiB");
  JVal doc;
  if (!Reader(text, len).parse(&doc, err)) return OVL_E_ARG;
  if (doc.kind != JVal::kObj) return bad(err, OVL_E_ARG, "manifest must be a JSON object");
  std::string key;
  if (!only_keys(doc, {"base_model_hash", "quantization", "runtime", "mode", "tokenizer_id", "timestamp_utc",
                       "adapters"}, &key))
    return bad(err, OVL_E_ARG, "unknown manifest field \"" + key + "\"");
  Manifest m;
  if (!parse_hash(doc.get("base_model_hash"), m.base_hash))
    return bad(err, OVL_E_ARG, "base_model_hash must be \"sha256:\" and 64 lowercase hex digits");
  const JVal* q = doc.get("quantization");
  if (!q || q->kind != JVal::kStr) return bad(err, OVL_E_ARG, "quantization must be a string");
  if (q->s == "q8_0") m.quant = OVL_Q8_0;
  else if (q->s == "q4_0") m.quant = OVL_Q4_0;
  else if (q->s == "q4_K") m.quant = OVL_Q4_K;
  else return bad(err, OVL_E_QUANT, "unsupported quantization profile \"" + q->s + "\"");
  for (const char* k : {"tokenizer_id", "timestamp_utc"})
    if (const JVal* v = doc.get(k))
      if (v->kind != JVal::kStr) return bad(err, OVL_E_ARG, std::string(k) + " must be a string");
  m.mode = OVL_MODE_STACK;
  if (const JVal* v = doc.get("mode")) {
    if (v->kind == JVal::kStr && v->s == "stack") m.mode = OVL_MODE_STACK;
    else if (v->kind == JVal::kStr && v->s == "table") m.mode = OVL_MODE_TABLE;
    else return bad(err, OVL_E_ARG, "mode must be \"stack\" or \"table\"");
  }
  if (const JVal* r = doc.get("runtime")) {
    if (r->kind != JVal::kObj || !only_keys(*r, {"name", "version"}, &key))
      return bad(err, OVL_E_ARG, "runtime must be an object with name and version");
    const JVal* nm = r->get("name");
    const JVal* ver = r->get("version");
    if (!nm || !ver || nm->kind != JVal::kStr || ver->kind != JVal::kStr)
      return bad(err, OVL_E_ARG, "runtime must be an object with name and version");
    if (nm->s != kManifestRuntimeName || ver->s != kManifestRuntimeVersion)
      return bad(err, OVL_E_ARG, "runtime " + nm->s + " " + ver->s + " is not this library (" +
                                     kManifestRuntimeName + " " + kManifestRuntimeVersion + ")");
  }
  const JVal* ads = doc.get("adapters");
  if (!ads || ads->kind != JVal::kArr) return bad(err, OVL_E_ARG, "adapters must be an array");
  if (ads->arr.size() > static_cast<size_t>(OVL_MAX_TABLE)) return bad(err, OVL_E_ARG, "too many adapters");
  for (size_t i = 0; i < ads->arr.size(); ++i) {
    const JVal& a = ads->arr[i];
    const std::string at = "adapters[" + std::to_string(i) + "]";
    if (a.kind != JVal::kObj) return bad(err, OVL_E_ARG, at + " must be an object");
    if (!only_keys(a, {"name", "file_hash", "load_order", "merge_weight", "type", "rank", "required_base_hash",
                       "targets"}, &key))
      return bad(err, OVL_E_ARG, "unknown field \"" + key + "\" in " + at);
    ManifestAdapter e;
    const JVal* nm = a.get("name");
    if (!nm || nm->kind != JVal::kStr || nm->s.empty() || nm->s.size() > 63)
      return bad(err, OVL_E_ARG, at + ".name must be a string of 1 to 63 bytes");
    e.name = nm->s;
    if (!parse_hash(a.get("file_hash"), e.file_hash))
      return bad(err, OVL_E_ARG, at + ".file_hash must be \"sha256:\" and 64 lowercase hex digits");
    int64_t lo = 0;
    if (!parse_int(a.get("load_order"), 1, 0x7FFFFFFF, &lo))
      return bad(err, OVL_E_ARG, at + ".load_order must be an integer from 1 to 2^31-1");
    e.load_order = static_cast<uint32_t>(lo);
    const JVal* w = a.get("merge_weight");
    if (!w || w->kind != JVal::kNum) return bad(err, OVL_E_ARG, at + ".merge_weight must be a number");
    e.merge_weight = static_cast<float>(std::strtod(w->s.c_str(), nullptr));
    if (!std::isfinite(e.merge_weight)) return bad(err, OVL_E_ARG, at + ".merge_weight is not finite in binary32");
    e.type = OVL_ADAPTER_LORA;
    if (const JVal* t = a.get("type")) {
      if (t->kind == JVal::kStr && t->s == "lora") e.type = OVL_ADAPTER_LORA;
      else if (t->kind == JVal::kStr && t->s == "sparse") e.type = OVL_ADAPTER_SPARSE;
      else return bad(err, OVL_E_ARG, at + ".type must be \"lora\" or \"sparse\"");
    }
    if (const JVal* r = a.get("rank")) {
      int64_t rv = 0;
      if (e.type != OVL_ADAPTER_LORA || !parse_int(r, 1, OVL_MAX_RANK, &rv))
        return bad(err, OVL_E_ARG, at + ".rank must be an integer from 1 to OVL_MAX_RANK (low-rank adapters)");
      e.rank = static_cast<uint32_t>(rv);
    }
    if (a.get("required_base_hash")) {
      if (!parse_hash(a.get("required_base_hash"), e.required_base))
        return bad(err, OVL_E_ARG, at + ".required_base_hash must be \"sha256:\" and 64 lowercase hex digits");
      e.has_required_base = true;
    }
    if (const JVal* tg = a.get("targets")) {
      if (tg->kind != JVal::kArr) return bad(err, OVL_E_ARG, at + ".targets must be an array of tensor indices");
      for (const JVal& x : tg->arr) {
        int64_t ti = 0;
        if (!parse_int(&x, 0, 0x7FFFFFFF, &ti)) return bad(err, OVL_E_ARG, at + ".targets must hold tensor indices");
        e.targets.push_back(static_cast<uint32_t>(ti));
      }
      e.has_targets = true;
    }
    for (const ManifestAdapter& o : m.adapters) {
      if (o.name == e.name) return bad(err, OVL_E_DUPLICATE, at + " repeats the name \"" + e.name + "\"");
      if (std::memcmp(o.file_hash, e.file_hash, 32) == 0) return bad(err, OVL_E_DUPLICATE, at + " repeats a file_hash");
      if (o.load_order == e.load_order)
        return bad(err, OVL_E_ARG, at + " repeats load_order " + std::to_string(e.load_order) + ": the order is ambiguous");
    }
    m.adapters.push_back(std::move(e));
  }
  // increasing load_order (insertion sort: at most OVL_MAX_TABLE entries)
  for (size_t i = 1; i < m.adapters.size(); ++i)
    for (size_t j = i; j > 0 && m.adapters[j].load_order < m.adapters[j - 1].load_order; --j)
      std::swap(m.adapters[j], m.adapters[j - 1]);
  *out = std::move(m);
  err->clear();
  return OVL_OK;
}

}  // namespace ovl

extern "C" ovl_status ovl_manifest_parse(const char* text, size_t len, ovl_manifest* out) {
  using namespace ovl;
  Manifest m;
  std::string err;
  const ovl_status st = parse_manifest(text, len, &m, &err);
  set_context_free_error(err);
  if (st != OVL_OK || !out) return st != OVL_OK ? st : OVL_E_ARG;
  std::memset(out, 0, sizeof(*out));
  std::memcpy(out->base_digest, m.base_hash, 32);
  out->quant = m.quant;
  out->mode = m.mode;
  out->n_adapters = static_cast<uint32_t>(m.adapters.size());
  for (size_t i = 0; i < m.adapters.size(); ++i) {
    const ManifestAdapter& e = m.adapters[i];
    ovl_manifest_entry& d = out->adapters[i];
    std::memcpy(d.file_digest, e.file_hash, 32);
    d.type = e.type;
    d.load_order = e.load_order;
    d.merge_weight = e.merge_weight;
    d.rank = e.rank;
    d.n_targets = static_cast<uint32_t>(e.targets.size());
    d.has_required_base = e.has_required_base ? 1u : 0u;
    std::memcpy(d.required_base_digest, e.required_base, 32);
    std::strncpy(d.name, e.name.c_str(), sizeof(d.name) - 1);
  }
  return OVL_OK;
}
