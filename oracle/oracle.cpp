// CPU oracle for one functional training step given as a static op list.
//
// TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
// load this file; only the tests, the smoke check and the benchmark's CPU
// baseline use it.  It shares no code, header or table with the CUDA path.
//
// It is a plain, slow interpreter of the op semantics that trainkernel's code
// generator gives each operation (page "trainkernel 0.1.0 --
// trainkernel/codegen.py"):
//   * every tensor value is held after rounding to its dtype, and inputs are
//     widened exactly (`_round`, `read`);
//   * pointwise ops are evaluated in float32, one IEEE operation at a time
//     (the runtime compiles with --fmad=false, page "trainkernel/runtime.py",
//     `compile_program`), then rounded once to the op's output dtype
//     (`point_expr`, `store`);
//   * scalars enter as float32 literals (`_literal`);
//   * broadcasting is right-aligned and size-1 dimensions read index 0
//     (`operand`);
//   * mm/addmm accumulate sum_k a[r,k]*b[k,c]; the accumulator is a float32
//     value and addmm applies alpha*acc + beta*bias with the special cases
//     alpha == beta == 0, beta == 0 and alpha == 0 (`emit_mm`, `epilogue`);
//   * sum/mean reduce over `dims` (default: all, negative dims modulo rank)
//     and mean divides the float32 sum by float32(size); an empty mean is NaN
//     (`emit_reduction`).
// Readings where the pages leave freedom: the dot products and the sums are
// accumulated in double and rounded once to float32 (the GPU accumulates in
// float32 in its own order; the tests bound that difference); float64 tensors
// are an oracle-only dtype used to take finite-difference gradients, for
// which every op runs in double with no rounding.
//
// Rounding to bfloat16/float16 is round-to-nearest, ties to even, written from
// the definition in IEEE 754-2019 section 4.3.1: with p significand bits and
// minimum normal exponent emin, the quantum of |v| is 2^(max(e, emin) - p + 1)
// where 2^e <= |v| < 2^(e+1); the result is the nearest multiple of the
// quantum (ties to the even multiple), and a result beyond the largest finite
// value overflows to infinity.  NaN stays NaN and the sign of zero is kept.
#include <algorithm>
#include <cerrno>
#include <cfenv>
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <sstream>
#include <stdexcept>
#include <string>
#include <vector>
#ifdef _OPENMP
#include <omp.h>
#endif

namespace {

enum DType { F32 = 0, F16 = 1, BF16 = 2, F64 = 3 };

DType parse_dtype(const std::string& s) {
  if (s == "float32") return F32;
  if (s == "float16") return F16;
  if (s == "bfloat16") return BF16;
  if (s == "float64") return F64;
  throw std::runtime_error("oracle: unknown dtype " + s);
}

double round_format(double v, int p, int emin, double max_finite) {
  if (std::isnan(v) || std::isinf(v) || v == 0.0) return v;
  double a = std::fabs(v);
  int e2 = 0;
  std::frexp(a, &e2);              // a = f * 2^e2 with f in [0.5, 1)
  int e = std::max(e2 - 1, emin);  // 2^(e2-1) <= a < 2^e2
  double q = std::ldexp(1.0, e - (p - 1));
  double r = std::nearbyint(a / q) * q;  // default mode: to nearest, ties to even
  if (r > max_finite) r = INFINITY;
  return std::copysign(r, v);
}

double round_to(double v, DType dt) {
  switch (dt) {
    case F32: return static_cast<double>(static_cast<float>(v));
    case BF16: return round_format(v, 8, -126, std::ldexp(255.0, 120));
    case F16: return round_format(v, 11, -14, 65504.0);
    case F64: return v;
  }
  return v;
}

struct Spec {
  std::string buf;
  DType dt = F32;
  std::vector<int64_t> shape, strides;
  int64_t offset = 0;
  int64_t numel() const {
    int64_t n = 1;
    for (auto s : shape) n *= s;
    return n;
  }
  bool contiguous() const {
    int64_t st = 1;
    for (int d = int(shape.size()) - 1; d >= 0; --d) {
      if (shape[d] != 1 && strides[d] != st) return false;
      st *= shape[d];
    }
    return offset == 0;
  }
};

struct Operand {
  bool scalar = false;
  double value = 0.0;
  Spec t;
};

struct Op {
  std::string kind, name;
  std::vector<Operand> in;
  Spec out;
  double alpha = 1, beta = 1, threshold = 0, exponent = 2, value = 0;
  bool has_exponent = false;
  bool has_value = false;
  int ndims = -1;  // -1: reduce over every dim
  std::vector<int64_t> dims;
};

struct Program {
  std::vector<Spec> inputs, outputs;
  std::vector<Op> ops;
  std::map<std::string, std::vector<double>> buffers;
};

// ------------------------------------------------------------------ parsing

struct Reader {
  std::istringstream in;
  explicit Reader(const char* text) : in(text) {}
  std::string word() {
    std::string w;
    if (!(in >> w)) throw std::runtime_error("oracle: truncated program text");
    return w;
  }
  int64_t integer() { return std::stoll(word()); }
  double real() {
    std::string w = word();
    errno = 0;
    char* end = nullptr;
    double v = std::strtod(w.c_str(), &end);
    if (end == w.c_str()) throw std::runtime_error("oracle: bad number " + w);
    return v;
  }
  void expect(const char* tag) {
    std::string w = word();
    if (w != tag) throw std::runtime_error(std::string("oracle: expected ") + tag + ", got " + w);
  }
  Spec spec() {
    Spec s;
    s.buf = word();
    s.dt = parse_dtype(word());
    int64_t rank = integer();
    if (rank < 0 || rank > 8) throw std::runtime_error("oracle: bad rank");
    s.shape.resize(rank);
    s.strides.resize(rank);
    for (auto& v : s.shape) v = integer();
    for (auto& v : s.strides) v = integer();
    s.offset = integer();
    return s;
  }
};

Program parse(const char* text) {
  Reader r(text);
  Program p;
  r.expect("TKORACLE");
  r.expect("1");
  r.expect("INPUTS");
  int64_t n = r.integer();
  for (int64_t i = 0; i < n; ++i) p.inputs.push_back(r.spec());
  r.expect("OPS");
  n = r.integer();
  for (int64_t i = 0; i < n; ++i) {
    Op op;
    r.expect("OP");
    op.kind = r.word();
    op.name = r.word();
    int64_t k = r.integer();
    for (int64_t j = 0; j < k; ++j) {
      Operand o;
      std::string tag = r.word();
      if (tag == "S") {
        o.scalar = true;
        o.value = r.real();
      } else if (tag == "T") {
        o.t = r.spec();
      } else {
        throw std::runtime_error("oracle: bad operand tag " + tag);
      }
      op.in.push_back(o);
    }
    r.expect("OUT");
    op.out = r.spec();
    r.expect("ATTR");
    op.alpha = r.real();
    op.beta = r.real();
    op.threshold = r.real();
    op.exponent = r.real();
    op.value = r.real();
    op.has_exponent = r.integer() != 0;
    op.has_value = r.integer() != 0;
    op.ndims = int(r.integer());
    for (int j = 0; j < op.ndims; ++j) op.dims.push_back(r.integer());
    p.ops.push_back(op);
  }
  r.expect("OUTPUTS");
  n = r.integer();
  for (int64_t i = 0; i < n; ++i) p.outputs.push_back(r.spec());
  r.expect("END");
  return p;
}

// ---------------------------------------------------------------- reading

const std::vector<double>& storage(const Program& p, const std::string& buf) {
  auto it = p.buffers.find(buf);
  if (it == p.buffers.end()) throw std::runtime_error("oracle: buffer " + buf + " has no value");
  return it->second;
}

// A view bound to the values of its buffer.
struct View {
  const Spec* s = nullptr;
  const double* data = nullptr;
  int64_t size = 0;
};

View bind(const Program& p, const Spec& s) {
  const auto& v = storage(p, s.buf);
  return View{&s, v.data(), int64_t(v.size())};
}

// Element of a view at the given coordinates of its own shape.
double at(const View& v, const int64_t* coord) {
  int64_t idx = v.s->offset;
  for (size_t d = 0; d < v.s->shape.size(); ++d) idx += coord[d] * v.s->strides[d];
  if (idx < 0 || idx >= v.size) throw std::runtime_error("oracle: read out of bounds in " + v.s->buf);
  return v.data[idx];
}

void unravel(int64_t i, const std::vector<int64_t>& shape, int64_t* coord) {
  for (int d = int(shape.size()) - 1; d >= 0; --d) {
    int64_t n = std::max<int64_t>(shape[d], 1);
    coord[d] = i % n;
    i /= n;
  }
}

// An operand of an op: a float32/float64 literal or a bound tensor view.
struct Arg {
  bool scalar = false;
  double value = 0.0;
  View v;
};

std::vector<Arg> bind_args(const Program& p, const Op& op) {
  std::vector<Arg> args;
  for (const auto& o : op.in) {
    Arg a;
    a.scalar = o.scalar;
    a.value = o.value;
    if (!o.scalar) a.v = bind(p, o.t);
    args.push_back(a);
  }
  return args;
}

// Operand value at output element `i`: right-aligned broadcast, size-1 dims read 0.
double operand_at(const Arg& a, const Spec& out, int64_t i) {
  if (a.scalar) return a.value;
  const Spec& t = *a.v.s;
  int64_t oc[8], tc[8];
  unravel(i, out.shape, oc);
  size_t ro = out.shape.size(), rt = t.shape.size();
  if (rt > ro) throw std::runtime_error("oracle: invalid broadcast rank");
  for (size_t d = 0; d < rt; ++d) {
    int64_t od = t.shape[d], want = out.shape[d + ro - rt];
    if (od != 1 && od != want) throw std::runtime_error("oracle: incompatible broadcast dimensions");
    tc[d] = (od == 1) ? 0 : oc[d + ro - rt];
  }
  return at(a.v, tc);
}

// ------------------------------------------------------------ evaluation

template <typename T>
T pointwise(const Op& op, const T* v) {
  const std::string& k = op.kind;
  if (k == "add") { T t = T(op.alpha) * v[1]; return v[0] + t; }
  if (k == "sub") { T t = T(op.alpha) * v[1]; return v[0] - t; }
  if (k == "mul") return v[0] * v[1];
  if (k == "div") return v[0] / v[1];
  if (k == "neg") return -v[0];
  if (k == "relu") return v[0] < T(0) ? T(0) : v[0];
  if (k == "pow") {
    double e = op.in.size() > 1 ? op.in[1].value : op.exponent;
    if (e == 2.0) return v[0] * v[0];
    return std::pow(v[0], T(e));
  }
  if (k == "threshold_backward") return v[1] <= T(op.threshold) ? T(0) : v[0];
  // full: the value attribute when given, else the scalar operand, else 0
  // (page "trainkernel/codegen.py", point_expr)
  if (k == "full") return T(op.has_value ? op.value : op.in.empty() ? 0.0 : op.in[0].value);
  if (k == "cast") return v[0];
  throw std::runtime_error("oracle: unsupported pointwise op " + k);
}

bool is_pointwise(const std::string& k) {
  static const char* names[] = {"add", "sub", "mul", "div", "neg", "relu", "pow",
                                "threshold_backward", "full", "cast"};
  for (auto n : names) if (k == n) return true;
  return false;
}

// Number of leading operands a pointwise op reads as values.
size_t value_operands(const Op& op) {
  if (op.kind == "full") return 0;
  if (op.kind == "pow") {
    if (op.in.size() > 1 && !op.in[1].scalar) throw std::runtime_error("oracle: pow exponent must be a scalar");
    return 1;
  }
  if (op.kind == "neg" || op.kind == "relu" || op.kind == "cast") return 1;
  return 2;
}

// One output element of a pointwise op, computed in T and rounded.
template <typename T>
double pointwise_element(const Op& op, const std::vector<Arg>& args, int64_t i) {
  T v[3] = {T(0), T(0), T(0)};
  size_t n = value_operands(op);
  if (args.size() < n) throw std::runtime_error("oracle: too few operands for " + op.kind);
  for (size_t j = 0; j < n; ++j) v[j] = T(operand_at(args[j], op.out, i));
  return round_to(double(pointwise<T>(op, v)), op.out.dt);
}

struct MM {
  const Arg* a;
  const Arg* b;
  const Arg* bias;
  int64_t m, k, n;
};

MM matmul_operands(const Op& op, const std::vector<Arg>& args) {
  MM g{};
  size_t base = op.kind == "addmm" ? 1 : 0;
  if (args.size() < base + 2 || args[base].scalar || args[base + 1].scalar)
    throw std::runtime_error("oracle: mm requires two tensor operands");
  g.a = &args[base];
  g.b = &args[base + 1];
  g.bias = op.kind == "addmm" ? &args[0] : nullptr;
  const Spec& A = *g.a->v.s;
  const Spec& B = *g.b->v.s;
  if (A.shape.size() != 2 || B.shape.size() != 2 || A.shape[1] != B.shape[0])
    throw std::runtime_error("oracle: mm requires compatible rank-two tensors");
  g.m = A.shape[0];
  g.k = A.shape[1];
  g.n = B.shape[1];
  if (op.out.shape.size() != 2 || op.out.shape[0] != g.m || op.out.shape[1] != g.n)
    throw std::runtime_error("oracle: matrix output shape does not match its inputs");
  return g;
}

// One element (r, c) of mm/addmm; `absdot` receives sum_k |a[r,k] b[k,c]|.
template <typename T>
double matmul_element(const Op& op, const MM& g, int64_t i, double* absdot) {
  int64_t r = i / std::max<int64_t>(g.n, 1), c = i % std::max<int64_t>(g.n, 1);
  double acc = 0.0, mag = 0.0;
  for (int64_t kk = 0; kk < g.k; ++kk) {
    int64_t ca[2] = {r, kk}, cb[2] = {kk, c};
    double prod = at(g.a->v, ca) * at(g.b->v, cb);  // exact: a product of two floats
    acc += prod;
    mag += std::fabs(prod);
  }
  if (absdot) *absdot = mag;
  T accT = T(acc);
  T value = accT;
  if (op.kind == "addmm") {
    if (op.alpha == 0.0 && op.beta == 0.0) {
      value = T(0);
    } else if (op.beta == 0.0) {
      value = T(op.alpha) * accT;
    } else {
      T bias = T(operand_at(*g.bias, op.out, i));
      if (op.alpha == 0.0) {
        value = T(op.beta) * bias;
      } else {
        T s1 = T(op.alpha) * accT;
        T s2 = T(op.beta) * bias;
        value = s1 + s2;
      }
    }
  }
  return round_to(double(value), op.out.dt);
}

struct Red {
  std::vector<int> kept, reduced;
  std::vector<int64_t> kept_shape, red_shape;
  int64_t size = 1;
};

Red reduction_axes(const Op& op, const std::vector<Arg>& args) {
  if (args.empty() || args[0].scalar) throw std::runtime_error("oracle: reduction requires a tensor");
  const Spec& s = *args[0].v.s;
  int rank = int(s.shape.size());
  std::vector<bool> red(rank, false);
  if (op.ndims < 0) {
    for (int d = 0; d < rank; ++d) red[d] = true;
  } else {
    for (auto d : op.dims) {
      if (rank == 0) break;
      int64_t m = ((d % rank) + rank) % rank;
      red[m] = true;
    }
  }
  Red R;
  for (int d = 0; d < rank; ++d) {
    if (red[d]) { R.reduced.push_back(d); R.red_shape.push_back(s.shape[d]); R.size *= s.shape[d]; }
    else { R.kept.push_back(d); R.kept_shape.push_back(s.shape[d]); }
  }
  int64_t kept_n = 1;
  for (auto v : R.kept_shape) kept_n *= v;
  if (kept_n != op.out.numel()) throw std::runtime_error("oracle: reduction output shape does not match its axes");
  return R;
}

template <typename T>
double reduction_element(const Op& op, const std::vector<Arg>& args, const Red& R, int64_t row, double* absbound) {
  int64_t kc[8], rc[8], sc[8];
  unravel(row, R.kept_shape, kc);
  for (size_t j = 0; j < R.kept.size(); ++j) sc[R.kept[j]] = kc[j];
  double acc = 0.0, mag = 0.0;
  for (int64_t r = 0; r < R.size; ++r) {
    unravel(r, R.red_shape, rc);
    for (size_t j = 0; j < R.reduced.size(); ++j) sc[R.reduced[j]] = rc[j];
    double v = at(args[0].v, sc);
    acc += v;
    mag += std::fabs(v);
  }
  if (absbound) *absbound = mag;
  T accT = T(acc);
  T value = accT;
  if (op.kind == "mean") value = R.size ? accT / T(double(R.size)) : T(NAN);
  return round_to(double(value), op.out.dt);
}

// An op with its operands bound, ready to produce output elements.
struct Bound {
  const Op* op;
  std::vector<Arg> args;
  int kind;  // 0 pointwise, 1 matmul, 2 reduction
  MM mm{};
  Red red;
  bool wide;  // float64 arithmetic
};

Bound bind_op(const Program& p, const Op& op) {
  Bound b;
  b.op = &op;
  b.args = bind_args(p, op);
  b.wide = op.out.dt == F64;
  if (is_pointwise(op.kind)) {
    b.kind = 0;
    value_operands(op);
  } else if (op.kind == "mm" || op.kind == "addmm") {
    b.kind = 1;
    b.mm = matmul_operands(op, b.args);
  } else if (op.kind == "sum" || op.kind == "mean") {
    b.kind = 2;
    b.red = reduction_axes(op, b.args);
  } else {
    throw std::runtime_error("oracle: unsupported op " + op.kind);
  }
  return b;
}

double element(const Bound& b, int64_t i, double* bound) {
  if (bound) *bound = 0.0;
  const Op& op = *b.op;
  switch (b.kind) {
    case 0: return b.wide ? pointwise_element<double>(op, b.args, i) : pointwise_element<float>(op, b.args, i);
    case 1: return b.wide ? matmul_element<double>(op, b.mm, i, bound) : matmul_element<float>(op, b.mm, i, bound);
    default: return b.wide ? reduction_element<double>(op, b.args, b.red, i, bound)
                           : reduction_element<float>(op, b.args, b.red, i, bound);
  }
}

void eval_op(Program& p, const Op& op) {
  if (!op.out.contiguous()) throw std::runtime_error("oracle: op output must be a contiguous buffer: " + op.name);
  Bound b = bind_op(p, op);
  int64_t n = op.out.numel();
  std::vector<double> out(n);
  if (n > 0) element(b, 0, nullptr);  // surface shape errors before the parallel loop
  std::string err;
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t i = 0; i < n; ++i) {
    try {
      out[i] = element(b, i, nullptr);
    } catch (const std::exception& e) {
#pragma omp critical
      err = e.what();
    }
  }
  if (!err.empty()) throw std::runtime_error(err);
  p.buffers[op.out.buf] = std::move(out);
}

thread_local std::string g_error;

template <typename F>
int guarded(F&& f) {
  try {
    f();
    return 0;
  } catch (const std::exception& e) {
    g_error = e.what();
    return -1;
  }
}

}  // namespace

extern "C" {

const char* oracle_last_error(void) { return g_error.c_str(); }

int oracle_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void* oracle_load(const char* text) {
  try {
    std::fesetround(FE_TONEAREST);
    return new Program(parse(text));
  } catch (const std::exception& e) {
    g_error = e.what();
    return nullptr;
  }
}

void oracle_free(void* h) { delete static_cast<Program*>(h); }

int oracle_set(void* h, const char* buffer, const double* data, int64_t n) {
  return guarded([&] { static_cast<Program*>(h)->buffers[buffer].assign(data, data + n); });
}

int64_t oracle_size(void* h, const char* buffer) {
  auto* p = static_cast<Program*>(h);
  auto it = p->buffers.find(buffer);
  return it == p->buffers.end() ? -1 : int64_t(it->second.size());
}

int oracle_get(void* h, const char* buffer, double* out, int64_t n) {
  return guarded([&] {
    const std::string name(buffer);
    const auto& v = storage(*static_cast<Program*>(h), name);
    if (int64_t(v.size()) != n) throw std::runtime_error("oracle: size mismatch reading " + std::string(buffer));
    std::copy(v.begin(), v.end(), out);
  });
}

int oracle_run(void* h) {
  return guarded([&] {
    auto* p = static_cast<Program*>(h);
    for (const auto& op : p->ops) eval_op(*p, op);
  });
}

int oracle_eval_op(void* h, int index) {
  return guarded([&] {
    auto* p = static_cast<Program*>(h);
    if (index < 0 || index >= int(p->ops.size())) throw std::runtime_error("oracle: op index out of range");
    eval_op(*p, p->ops[index]);
  });
}

int oracle_eval_op_sampled(void* h, int index, const int64_t* idx, int64_t n, double* out, double* bound) {
  return guarded([&] {
    auto* p = static_cast<Program*>(h);
    if (index < 0 || index >= int(p->ops.size())) throw std::runtime_error("oracle: op index out of range");
    const Op& op = p->ops[index];
    Bound b = bind_op(*p, op);
    int64_t total = op.out.numel();
    for (int64_t j = 0; j < n; ++j)
      if (idx[j] < 0 || idx[j] >= total) throw std::runtime_error("oracle: sample index out of range");
    if (n > 0) element(b, idx[0], nullptr);
#pragma omp parallel for schedule(dynamic, 4)
    for (int64_t j = 0; j < n; ++j) out[j] = element(b, idx[j], bound ? bound + j : nullptr);
  });
}

// Output slot value: its view read from the buffer and rounded to its dtype.
int oracle_output(void* h, int slot, double* out, int64_t n) {
  return guarded([&] {
    auto* p = static_cast<Program*>(h);
    if (slot < 0 || slot >= int(p->outputs.size())) throw std::runtime_error("oracle: output slot out of range");
    const Spec& s = p->outputs[slot];
    if (s.numel() != n) throw std::runtime_error("oracle: output size mismatch");
    View v = bind(*p, s);
    int64_t c[8];
    for (int64_t i = 0; i < n; ++i) {
      unravel(i, s.shape, c);
      out[i] = round_to(at(v, c), s.dt);
    }
  });
}

int oracle_round(int dtype, const double* in, double* out, int64_t n) {
  return guarded([&] {
    if (dtype < 0 || dtype > 3) throw std::runtime_error("oracle: bad dtype code");
    for (int64_t i = 0; i < n; ++i) out[i] = round_to(in[i], DType(dtype));
  });
}

}  // extern "C"
