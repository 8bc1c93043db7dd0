// safetensors files of float32 tensors, host code. [LM4] "Build a language model in C# from
// scratch (4): running GPT-2 weights", "The safetensors format": an 8-byte little-endian header
// length N, N bytes of JSON mapping each tensor name to {dtype, shape, data_offsets [begin, end)}
// (offsets from the end of the header) plus an optional "__metadata__" object of strings, then
// the raw bytes. Only F32 is read; other dtypes are refused with GK_ERR_FORMAT.
//
// The writer lays tensors out back to back in the order given, pads the JSON with spaces to a
// multiple of 8 bytes and writes through a temporary file renamed into place, so a reader never
// sees a half-written file.
#include <fcntl.h>
#include <stdio.h>
#include <string.h>
#include <unistd.h>

#include <algorithm>
#include <string>
#include <utility>
#include <vector>

#include "common.cuh"

namespace {

thread_local std::string g_err;

gk_status st_fail(gk_status code, const std::string& msg) {
    g_err = msg;
    return code;
}

bool little_endian() {
    const uint16_t one = 1;
    return *reinterpret_cast<const uint8_t*>(&one) == 1;
}

// ---------------------------------------------------------------- a small JSON parser
struct Json {
    enum Kind { OBJ, ARR, STR, NUM, BOOL, NUL } kind = NUL;
    std::string str;
    bool is_int = false;
    int64_t ival = 0;
    std::vector<std::pair<std::string, Json>> obj;
    std::vector<Json> arr;
};

struct Parser {
    const char* p;
    const char* e;
    std::string err;

    void ws() {
        while (p < e && (*p == ' ' || *p == '\t' || *p == '\n' || *p == '\r')) ++p;
    }
    bool fail(const char* what) {
        if (err.empty()) err = what;
        return false;
    }
    static void put_utf8(std::string& s, uint32_t c) {
        if (c < 0x80) {
            s += (char)c;
        } else if (c < 0x800) {
            s += (char)(0xC0 | (c >> 6));
            s += (char)(0x80 | (c & 0x3F));
        } else if (c < 0x10000) {
            s += (char)(0xE0 | (c >> 12));
            s += (char)(0x80 | ((c >> 6) & 0x3F));
            s += (char)(0x80 | (c & 0x3F));
        } else {
            s += (char)(0xF0 | (c >> 18));
            s += (char)(0x80 | ((c >> 12) & 0x3F));
            s += (char)(0x80 | ((c >> 6) & 0x3F));
            s += (char)(0x80 | (c & 0x3F));
        }
    }
    // four hex digits of a \u escape
    bool hex4(uint32_t& v) {
        if (e - p < 4) return fail("short \\u escape");
        for (int k = 0; k < 4; ++k) {
            const char h = *p++;
            const int d = h >= '0' && h <= '9' ? h - '0'
                          : h >= 'a' && h <= 'f' ? h - 'a' + 10
                          : h >= 'A' && h <= 'F' ? h - 'A' + 10
                                                 : -1;
            if (d < 0) return fail("bad \\u escape");
            v = v * 16 + (uint32_t)d;
        }
        return true;
    }
    bool string(std::string& out) {
        if (p >= e || *p != '"') return fail("expected a string");
        ++p;
        while (p < e && *p != '"') {
            char c = *p++;
            if ((unsigned char)c < 0x20) return fail("control character in a string");
            if (c != '\\') {
                out += c;
                continue;
            }
            if (p >= e) return fail("unterminated escape");
            char x = *p++;
            switch (x) {
                case '"': out += '"'; break;
                case '\\': out += '\\'; break;
                case '/': out += '/'; break;
                case 'b': out += '\b'; break;
                case 'f': out += '\f'; break;
                case 'n': out += '\n'; break;
                case 'r': out += '\r'; break;
                case 't': out += '\t'; break;
                case 'u': {
                    uint32_t c4 = 0;
                    if (!hex4(c4)) return false;
                    if (c4 >= 0xD800 && c4 <= 0xDBFF) {  // a high surrogate: its low half must follow
                        uint32_t lo = 0;
                        if (e - p < 2 || p[0] != '\\' || p[1] != 'u') return fail("lone surrogate");
                        p += 2;
                        if (!hex4(lo)) return false;
                        if (lo < 0xDC00 || lo > 0xDFFF) return fail("lone surrogate");
                        c4 = 0x10000 + ((c4 - 0xD800) << 10) + (lo - 0xDC00);
                    } else if (c4 >= 0xDC00 && c4 <= 0xDFFF) {
                        return fail("lone surrogate");
                    }
                    put_utf8(out, c4);
                    break;
                }
                default: return fail("bad escape");
            }
        }
        if (p >= e) return fail("unterminated string");
        ++p;
        return true;
    }
    bool number(Json& v) {
        const char* s = p;
        bool neg = false, frac = false;
        if (p < e && *p == '-') {
            neg = true;
            ++p;
        }
        int64_t acc = 0;
        bool overflow = false, digits = false;
        while (p < e && *p >= '0' && *p <= '9') {
            digits = true;
            if (acc > (INT64_MAX - 9) / 10) overflow = true;
            acc = acc * 10 + (*p++ - '0');
        }
        if (!digits) return fail("bad number");
        while (p < e && (*p == '.' || *p == 'e' || *p == 'E' || *p == '+' || *p == '-' || (*p >= '0' && *p <= '9'))) {
            frac = true;
            ++p;
        }
        v.kind = Json::NUM;
        v.is_int = !frac && !overflow;
        v.ival = neg ? -acc : acc;
        v.str.assign(s, p);
        return true;
    }
    bool literal(const char* word, Json::Kind k, Json& v) {
        size_t n = strlen(word);
        if ((size_t)(e - p) < n || strncmp(p, word, n) != 0) return fail("bad literal");
        p += n;
        v.kind = k;
        return true;
    }
    bool value(Json& v, int depth) {
        if (depth > 64) return fail("nesting too deep");
        ws();
        if (p >= e) return fail("unexpected end");
        switch (*p) {
            case '{': {
                ++p;
                v.kind = Json::OBJ;
                ws();
                if (p < e && *p == '}') {
                    ++p;
                    return true;
                }
                while (true) {
                    ws();
                    std::string key;
                    if (!string(key)) return false;
                    for (auto& kv : v.obj)
                        if (kv.first == key) return fail("duplicate key");
                    ws();
                    if (p >= e || *p != ':') return fail("expected ':'");
                    ++p;
                    Json child;
                    if (!value(child, depth + 1)) return false;
                    v.obj.emplace_back(std::move(key), std::move(child));
                    ws();
                    if (p < e && *p == ',') {
                        ++p;
                        continue;
                    }
                    if (p < e && *p == '}') {
                        ++p;
                        return true;
                    }
                    return fail("expected ',' or '}'");
                }
            }
            case '[': {
                ++p;
                v.kind = Json::ARR;
                ws();
                if (p < e && *p == ']') {
                    ++p;
                    return true;
                }
                while (true) {
                    Json child;
                    if (!value(child, depth + 1)) return false;
                    v.arr.push_back(std::move(child));
                    ws();
                    if (p < e && *p == ',') {
                        ++p;
                        continue;
                    }
                    if (p < e && *p == ']') {
                        ++p;
                        return true;
                    }
                    return fail("expected ',' or ']'");
                }
            }
            case '"': v.kind = Json::STR; return string(v.str);
            case 't': return literal("true", Json::BOOL, v);
            case 'f': return literal("false", Json::BOOL, v);
            case 'n': return literal("null", Json::NUL, v);
            default: return number(v);
        }
    }
};

// JSON text is UTF-8: well-formed sequences only (no overlongs, surrogates or code points past
// U+10FFFF)
bool valid_utf8(const std::string& t) {
    const unsigned char* p = reinterpret_cast<const unsigned char*>(t.data());
    const unsigned char* e = p + t.size();
    while (p < e) {
        const unsigned c = *p++;
        if (c < 0x80) continue;
        int more;
        unsigned cp;
        if (c >= 0xC2 && c <= 0xDF) {
            more = 1;
            cp = c & 0x1F;
        } else if (c >= 0xE0 && c <= 0xEF) {
            more = 2;
            cp = c & 0x0F;
        } else if (c >= 0xF0 && c <= 0xF4) {
            more = 3;
            cp = c & 0x07;
        } else {
            return false;
        }
        if (e - p < more) return false;
        for (int k = 0; k < more; ++k) {
            if ((p[k] & 0xC0) != 0x80) return false;
            cp = (cp << 6) | (p[k] & 0x3F);
        }
        p += more;
        if ((more == 2 && cp < 0x800) || (more == 3 && cp < 0x10000) || cp > 0x10FFFF || (cp >= 0xD800 && cp <= 0xDFFF))
            return false;
    }
    return true;
}

const Json* field(const Json& o, const char* key) {
    for (auto& kv : o.obj)
        if (kv.first == key) return &kv.second;
    return nullptr;
}

void json_escape(std::string& out, const std::string& s) {
    out += '"';
    for (unsigned char c : s) {
        if (c == '"' || c == '\\') {
            out += '\\';
            out += (char)c;
        } else if (c < 0x20) {
            char buf[8];
            snprintf(buf, sizeof buf, "\\u%04x", c);
            out += buf;
        } else {
            out += (char)c;
        }
    }
    out += '"';
}

constexpr size_t CHUNK = 64u << 20;  // host staging for device transfers and large reads

}  // namespace

struct gk_st {
    struct Entry {
        std::string name, dtype;
        std::vector<int64_t> shape;
        int64_t begin = 0, end = 0;
    };
    std::string path;
    int64_t data_start = 0;
    std::vector<Entry> entries;
    std::vector<std::pair<std::string, std::string>> meta;
};

extern "C" {

const char* gk_st_last_error(void) { return g_err.c_str(); }

gk_status gk_st_open(const char* path, gk_st** out) {
    if (!path || !out) return st_fail(GK_ERR_ARG, "gk_st_open: null argument");
    *out = nullptr;
    if (!little_endian()) return st_fail(GK_ERR_UNSUPPORTED, "gk_st_open: big-endian host");
    FILE* f = fopen(path, "rb");
    if (!f) return st_fail(GK_ERR_IO, std::string("gk_st_open: cannot open ") + path);
    uint8_t lb[8];
    int64_t size = -1;
    if (fseeko(f, 0, SEEK_END) == 0) size = (int64_t)ftello(f);
    if (size < 8 || fseeko(f, 0, SEEK_SET) != 0 || fread(lb, 1, 8, f) != 8) {
        fclose(f);
        return st_fail(GK_ERR_FORMAT, "gk_st_open: shorter than the 8-byte header length");
    }
    uint64_t n = 0;
    for (int k = 7; k >= 0; --k) n = (n << 8) | lb[k];
    if (n > (uint64_t)(size - 8) || n > (1ull << 30)) {
        fclose(f);
        return st_fail(GK_ERR_FORMAT, "gk_st_open: header length past the end of the file");
    }
    std::string text(n, '\0');
    if (n && fread(&text[0], 1, n, f) != n) {
        fclose(f);
        return st_fail(GK_ERR_IO, "gk_st_open: short read of the header");
    }
    fclose(f);
    if (!valid_utf8(text)) return st_fail(GK_ERR_FORMAT, "gk_st_open: header is not valid UTF-8");
    Parser ps{text.data(), text.data() + text.size(), {}};
    Json root;
    bool ok = ps.value(root, 0);
    ps.ws();
    if (!ok || ps.p != ps.e) return st_fail(GK_ERR_FORMAT, "gk_st_open: header JSON: " + (ps.err.empty() ? std::string("trailing data") : ps.err));
    if (root.kind != Json::OBJ) return st_fail(GK_ERR_FORMAT, "gk_st_open: header is not a JSON object");
    gk_st* st = new gk_st();
    st->path = path;
    st->data_start = 8 + (int64_t)n;
    auto bad = [&](const std::string& m) {
        delete st;
        return st_fail(GK_ERR_FORMAT, "gk_st_open: " + m);
    };
    for (auto& kv : root.obj) {
        const Json& v = kv.second;
        if (kv.first == "__metadata__") {
            if (v.kind != Json::OBJ) return bad("__metadata__ is not an object");
            for (auto& m : v.obj) {
                if (m.second.kind != Json::STR) return bad("__metadata__ value of " + m.first + " is not a string");
                st->meta.emplace_back(m.first, m.second.str);
            }
            continue;
        }
        const Json *dt = v.kind == Json::OBJ ? field(v, "dtype") : nullptr, *sh = v.kind == Json::OBJ ? field(v, "shape") : nullptr,
                   *off = v.kind == Json::OBJ ? field(v, "data_offsets") : nullptr;
        if (!dt || dt->kind != Json::STR || !sh || sh->kind != Json::ARR || !off || off->kind != Json::ARR ||
            off->arr.size() != 2)
            return bad(kv.first + ": needs dtype, shape and data_offsets");
        gk_st::Entry e;
        e.name = kv.first;
        e.dtype = dt->str;
        // the element count times 4 bytes must stay within int64: a product that wrapped could
        // otherwise match data_offsets for a nonsensical shape
        int64_t count = 1;
        for (auto& d : sh->arr) {
            if (d.kind != Json::NUM || !d.is_int || d.ival < 0) return bad(kv.first + ": bad shape");
            if (d.ival > 0 && count > (INT64_MAX / 4) / d.ival) return bad(kv.first + ": shape too large");
            count *= d.ival;
            e.shape.push_back(d.ival);
        }
        for (auto& o : off->arr)
            if (o.kind != Json::NUM || !o.is_int || o.ival < 0) return bad(kv.first + ": bad data_offsets");
        e.begin = off->arr[0].ival;
        e.end = off->arr[1].ival;
        if (e.end < e.begin || e.end > size - st->data_start) return bad(kv.first + ": data_offsets outside the file");
        st->entries.push_back(std::move(e));
    }
    *out = st;
    return GK_OK;
}

void gk_st_close(gk_st* st) { delete st; }

int gk_st_count(const gk_st* st) { return st ? (int)st->entries.size() : -1; }

const char* gk_st_name(const gk_st* st, int i) {
    return st && i >= 0 && i < (int)st->entries.size() ? st->entries[i].name.c_str() : nullptr;
}

const char* gk_st_dtype(const gk_st* st, int i) {
    return st && i >= 0 && i < (int)st->entries.size() ? st->entries[i].dtype.c_str() : nullptr;
}

int gk_st_ndim(const gk_st* st, int i) {
    return st && i >= 0 && i < (int)st->entries.size() ? (int)st->entries[i].shape.size() : -1;
}

const int64_t* gk_st_shape(const gk_st* st, int i) {
    return st && i >= 0 && i < (int)st->entries.size() ? st->entries[i].shape.data() : nullptr;
}

int gk_st_find(const gk_st* st, const char* name) {
    if (!st || !name) return -1;
    for (size_t i = 0; i < st->entries.size(); ++i)
        if (st->entries[i].name == name) return (int)i;
    return -1;
}

const char* gk_st_metadata(const gk_st* st, const char* key) {
    if (!st || !key) return nullptr;
    for (auto& m : st->meta)
        if (m.first == key) return m.second.c_str();
    return nullptr;
}

gk_status gk_st_read_f32(const gk_st* st, int i, float* dst, int64_t n, int dst_on_device) {
    if (!st || i < 0 || i >= (int)st->entries.size() || !dst || n < 0)
        return st_fail(GK_ERR_ARG, "gk_st_read_f32: bad argument");
    const gk_st::Entry& e = st->entries[i];
    if (e.dtype != "F32") return st_fail(GK_ERR_FORMAT, e.name + ": dtype " + e.dtype + ", only F32 is handled");
    int64_t count = 1;
    for (int64_t d : e.shape) count *= d;
    if (e.end - e.begin != 4 * count) return st_fail(GK_ERR_FORMAT, e.name + ": data_offsets do not match the shape");
    if (n != count) return st_fail(GK_ERR_ARG, e.name + ": destination size differs from the tensor's");
    const int fd = open(st->path.c_str(), O_RDONLY);
    if (fd < 0) return st_fail(GK_ERR_IO, "gk_st_read_f32: cannot open " + st->path);
    std::vector<char> stage(dst_on_device ? std::min<size_t>(CHUNK, (size_t)(4 * count)) : 0);
    int64_t done = 0, total = 4 * count;
    gk_status s = GK_OK;
    while (done < total && s == GK_OK) {
        const size_t want = dst_on_device ? std::min<size_t>(CHUNK, (size_t)(total - done)) : (size_t)(total - done);
        char* to = dst_on_device ? stage.data() : reinterpret_cast<char*>(dst) + done;
        size_t got = 0;
        while (got < want) {
            ssize_t r = pread(fd, to + got, std::min<size_t>(want - got, CHUNK), st->data_start + e.begin + done + got);
            if (r <= 0) {
                s = st_fail(GK_ERR_IO, e.name + ": short read");
                break;
            }
            got += (size_t)r;
        }
        if (s == GK_OK && dst_on_device &&
            cudaMemcpy(reinterpret_cast<char*>(dst) + done, stage.data(), want, cudaMemcpyHostToDevice) != cudaSuccess)
            s = st_fail(GK_ERR_CUDA, e.name + ": copy to the device failed");
        done += (int64_t)want;
    }
    close(fd);
    return s;
}

gk_status gk_st_write_f32(const char* path, int n, const char* const* names, const int* ndims, const int64_t* shapes,
                          const float* const* data, int data_on_device, int n_meta, const char* const* meta_keys,
                          const char* const* meta_values) {
    if (!path || n < 0 || (n > 0 && (!names || !ndims || !data)) || n_meta < 0 ||
        (n_meta > 0 && (!meta_keys || !meta_values)))
        return st_fail(GK_ERR_ARG, "gk_st_write_f32: bad argument");
    if (!little_endian()) return st_fail(GK_ERR_UNSUPPORTED, "gk_st_write_f32: big-endian host");
    std::string hdr = "{";
    if (n_meta > 0) {
        hdr += "\"__metadata__\":{";
        for (int k = 0; k < n_meta; ++k) {
            if (!meta_keys[k] || !meta_values[k]) return st_fail(GK_ERR_ARG, "gk_st_write_f32: null metadata");
            if (k) hdr += ',';
            json_escape(hdr, meta_keys[k]);
            hdr += ':';
            json_escape(hdr, meta_values[k]);
        }
        hdr += "}";
    }
    std::vector<int64_t> bytes(n);
    int64_t begin = 0, si = 0;
    for (int t = 0; t < n; ++t) {
        if (!names[t] || !*names[t] || !strcmp(names[t], "__metadata__") || ndims[t] < 0 || (ndims[t] && !shapes) ||
            (!data[t]))
            return st_fail(GK_ERR_ARG, "gk_st_write_f32: bad tensor " + std::to_string(t));
        for (int u = 0; u < t; ++u)
            if (!strcmp(names[u], names[t])) return st_fail(GK_ERR_ARG, std::string("gk_st_write_f32: duplicate name ") + names[t]);
        int64_t count = 1;
        std::string shp = "[";
        for (int d = 0; d < ndims[t]; ++d) {
            const int64_t v = shapes[si + d];
            if (v < 0) return st_fail(GK_ERR_ARG, std::string("gk_st_write_f32: negative extent in ") + names[t]);
            count *= v;
            if (d) shp += ',';
            shp += std::to_string(v);
        }
        shp += "]";
        si += ndims[t];
        bytes[t] = 4 * count;
        if (n_meta > 0 || t > 0) hdr += ',';
        json_escape(hdr, names[t]);
        hdr += ":{\"dtype\":\"F32\",\"shape\":" + shp + ",\"data_offsets\":[" + std::to_string(begin) + "," +
               std::to_string(begin + bytes[t]) + "]}";
        begin += bytes[t];
    }
    hdr += "}";
    hdr.append((8 - hdr.size() % 8) % 8, ' ');
    const std::string tmp = std::string(path) + ".tmp";
    FILE* f = fopen(tmp.c_str(), "wb");
    if (!f) return st_fail(GK_ERR_IO, "gk_st_write_f32: cannot create " + tmp);
    uint8_t lb[8];
    uint64_t len = hdr.size();
    for (int k = 0; k < 8; ++k) lb[k] = (uint8_t)(len >> (8 * k));
    bool ok = fwrite(lb, 1, 8, f) == 8 && fwrite(hdr.data(), 1, hdr.size(), f) == hdr.size();
    std::vector<char> stage(data_on_device ? CHUNK : 0);
    gk_status s = GK_OK;
    for (int t = 0; t < n && ok && s == GK_OK; ++t) {
        const char* src = reinterpret_cast<const char*>(data[t]);
        for (int64_t done = 0; done < bytes[t] && ok;) {
            const size_t w = std::min<size_t>(CHUNK, (size_t)(bytes[t] - done));
            const char* from = src + done;
            if (data_on_device) {
                if (cudaMemcpy(stage.data(), src + done, w, cudaMemcpyDeviceToHost) != cudaSuccess) {
                    s = st_fail(GK_ERR_CUDA, std::string(names[t]) + ": copy from the device failed");
                    break;
                }
                from = stage.data();
            }
            ok = fwrite(from, 1, w, f) == w;
            done += (int64_t)w;
        }
    }
    ok = (fclose(f) == 0) && ok;
    if (s == GK_OK && !ok) s = st_fail(GK_ERR_IO, "gk_st_write_f32: write to " + tmp + " failed");
    if (s == GK_OK && rename(tmp.c_str(), path) != 0) s = st_fail(GK_ERR_IO, std::string("gk_st_write_f32: cannot rename to ") + path);
    if (s != GK_OK) remove(tmp.c_str());
    return s;
}

}  // extern "C"
