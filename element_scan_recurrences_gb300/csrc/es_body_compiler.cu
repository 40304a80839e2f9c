// es_body_compiler.cu -- translate an element-scan body given as text into a
// CUDA functor (host code).
//
// What a body may contain: "Nonlinear element scans", "Arguments and body"
// (pointwise arithmetic, transcendental functions, comparisons, `where`,
// scalar constants, boolean intermediates, casts between f32 and bool; with
// `:state-axis` scalars and vectors of 1..16 values, `sum` and `max` reducing
// a vector, a one-value vector broadcasting against the state; a scalar
// state's body cannot reduce).  Operation names and the overloaded
// arithmetic: "Tensor operations" ("Shapes, dtypes, broadcasting" and
// "Operations": plain numbers mixed with a tensor become constants, plain
// numbers at the front of an n-ary `*` fold first).
//
// The body is traced once, as the pages describe: every operation on a
// tensor value appends one statement to the functor, every operation on
// plain numbers is done here in double precision, and a plain number meeting
// a tensor becomes the f32 constant nearest to it.  Each tensor statement is
// one f32 operation rounded to nearest: + - * / and sqrt are the IEEE
// operations (the _rn intrinsics, which also keep a multiply and an add from
// fusing), exp, log, tanh, sin, cos, acos, asin, atan2, pow and rsqrt are
// CUDA's f32 functions, `maximum` / `minimum` are IEEE 754-2019 (PTX
// max.NaN / min.NaN), comparisons are IEEE (false on NaN except !=).
// Readings of what the pages leave open: `max` with one tensor argument is the
// reduction (the elementwise pair is `maximum`); the comparisons are
// < <= > >= = !=; `and`, `or`, `not` combine booleans; (cast x :bool) is
// x != 0; `let` binds in order; a `sum` adds a thread's values in state order
// and then the lane's threads pairwise.
#include "es_body_compiler.h"

#include <cmath>
#include <cstdio>
#include <cstring>
#include <algorithm>
#include <cctype>
#include <map>
#include <set>
#include <sstream>

namespace es {
namespace body {
namespace {

[[noreturn]] void fail(const char* code, const std::string& msg) { throw Error{code, msg}; }

// ---------------------------------------------------------------------------
// reader

bool is_delim(char c) { return c == '(' || c == ')' || c == '[' || c == ']' || c == ';' || std::isspace((unsigned char)c); }

// [+-]? (digits [. digits*] | . digits) ([eE] [+-]? digits)?
bool parse_number(const std::string& t, double* out) {
    size_t i = 0;
    if (i < t.size() && (t[i] == '+' || t[i] == '-')) ++i;
    size_t int_digits = 0, frac_digits = 0;
    while (i < t.size() && std::isdigit((unsigned char)t[i])) ++i, ++int_digits;
    if (i < t.size() && t[i] == '.') {
        ++i;
        while (i < t.size() && std::isdigit((unsigned char)t[i])) ++i, ++frac_digits;
    }
    if (int_digits == 0 && frac_digits == 0) return false;
    if (i < t.size() && (t[i] == 'e' || t[i] == 'E')) {
        ++i;
        if (i < t.size() && (t[i] == '+' || t[i] == '-')) ++i;
        size_t exp_digits = 0;
        while (i < t.size() && std::isdigit((unsigned char)t[i])) ++i, ++exp_digits;
        if (exp_digits == 0) return false;
    }
    if (i != t.size()) return false;
    *out = std::strtod(t.c_str(), nullptr);   // correctly rounded to double
    return true;
}

class Reader {
public:
    explicit Reader(const std::string& text) : text_(text) {}

    Form read_all() {
        Form f = read();
        skip();
        if (pos_ != text_.size()) fail("parse", "text after the body");
        return f;
    }

private:
    void skip() {
        while (pos_ < text_.size()) {
            if (std::isspace((unsigned char)text_[pos_])) {
                ++pos_;
            } else if (text_[pos_] == ';') {
                while (pos_ < text_.size() && text_[pos_] != '\n') ++pos_;
            } else {
                break;
            }
        }
    }

    Form read() {
        skip();
        if (pos_ >= text_.size()) fail("parse", "unexpected end of body text");
        const char c = text_[pos_];
        if (c == '(' || c == '[') {
            const char close = c == '(' ? ')' : ']';
            ++pos_;
            Form f;
            f.kind = c == '(' ? Form::kList : Form::kVec;
            for (;;) {
                skip();
                if (pos_ >= text_.size()) fail("parse", std::string("missing '") + close + "'");
                if (text_[pos_] == close) {
                    ++pos_;
                    return f;
                }
                if (text_[pos_] == ')' || text_[pos_] == ']')
                    fail("parse", std::string("mismatched '") + text_[pos_] + "'");
                f.items.push_back(read());
            }
        }
        if (c == ')' || c == ']') fail("parse", std::string("unexpected '") + c + "'");
        const size_t start = pos_;
        while (pos_ < text_.size() && !is_delim(text_[pos_])) ++pos_;
        const std::string tok = text_.substr(start, pos_ - start);
        Form f;
        if (parse_number(tok, &f.num)) {
            f.kind = Form::kNum;
        } else if (tok == "true" || tok == "false") {
            f.kind = Form::kBool;
            f.b = tok == "true";
        } else if (tok[0] == ':') {
            f.kind = Form::kKw;
            f.s = tok;
        } else {
            f.kind = Form::kSym;
            f.s = tok;
        }
        return f;
    }

    const std::string& text_;
    size_t pos_ = 0;
};

// ---------------------------------------------------------------------------
// values while tracing

struct Val {
    enum Kind { kNumber, kBoolConst, kTensor } kind = kNumber;
    double num = 0.0;
    bool b = false;
    std::string name;     // tensor: an expression naming it (array name if wide)
    bool is_bool = false; // tensor dtype: bool or f32
    bool wide = false;    // tensor width: the state's W (array of E) or one
    bool diff = false;    // depends on the state or a sequence through differentiable operations
};

// One differentiable operation of the trace (the tape the VJP sweeps back).
struct Node {
    std::string op;
    Val out;
    std::vector<Val> args;
    Val mask;             // `where`'s condition
};

Val number(double v) {
    Val r;
    r.kind = Val::kNumber;
    r.num = v;
    return r;
}

Val bool_const(bool v) {
    Val r;
    r.kind = Val::kBoolConst;
    r.b = v;
    return r;
}

std::string f32_literal(double v) {
    const float f = static_cast<float>(v);   // round to nearest f32
    uint32_t bits;
    std::memcpy(&bits, &f, 4);
    char buf[64];
    std::snprintf(buf, sizeof(buf), "__uint_as_float(0x%08xu)", bits);
    return buf;
}

double num_max(double a, double b) { return (a >= b || std::isnan(a)) ? a : b; }

using Env = std::map<std::string, Val>;

class Tracer {
public:
    Tracer(int W, bool vector) : W_(W), vector_(vector) {}

    std::string code;

    Val eval(const Form& f, const Env& env);

    std::string ref(const Val& v) const {
        if (v.kind == Val::kNumber) return f32_literal(v.num);
        if (v.kind == Val::kBoolConst) return v.b ? "true" : "false";
        return v.wide ? v.name + "[e]" : v.name;
    }

    // a plain number meeting a tensor: an f32 (or bool) constant
    Val tensor(const Val& v) const {
        if (v.kind == Val::kTensor) return v;
        Val r;
        r.kind = Val::kTensor;
        r.is_bool = v.kind == Val::kBoolConst;
        r.name = ref(v);
        r.wide = false;
        return r;
    }

    Val f32(const Val& v, const std::string& what) const {
        Val t = tensor(v);
        if (t.is_bool) fail("E-DIM-002", what + " wants f32, got bool");
        return t;
    }

    Val boolean(const Val& v, const std::string& what) const {
        Val t = tensor(v);
        if (!t.is_bool) fail("E-DIM-002", what + " wants bool, got f32");
        return t;
    }

    // A statement computing a new value.  `op` names a differentiable
    // operation of `args` (recorded on the tape when one of them is
    // differentiable); without it the value has no gradient.
    Val emit(bool is_bool, bool wide, const std::string& expr, const char* op = nullptr,
             const std::vector<Val>& args = {}, const Val& mask = Val()) {
        Val r;
        r.kind = Val::kTensor;
        r.is_bool = is_bool;
        r.wide = wide;
        r.name = "v" + std::to_string(next_++);
        if (op != nullptr && !is_bool) {
            for (const Val& a : args) r.diff = r.diff || a.diff;
            if (r.diff) tape.push_back(Node{op, r, args, mask});
        }
        const char* type = is_bool ? "bool" : "float";
        std::string stmt;
        if (wide) {
            stmt = std::string("        ") + type + " " + r.name + "[E];\n#pragma unroll\n        for (int e = 0; e < E; ++e) " +
                   r.name + "[e] = " + expr + ";\n";
        } else {
            stmt = std::string("        const ") + type + " " + r.name + " = " + expr + ";\n";
        }
        code += stmt;
        stmts.push_back(Stmt{r.name, stmt, names_in(expr)});
        return r;
    }

    // one emitted statement: the value it defines, its text, the values and
    // arguments (`h`, `sw[k]`, `sn[k]`) its expression reads
    struct Stmt {
        std::string name;
        std::string code;
        std::vector<std::string> deps;
    };
    std::vector<Stmt> stmts;

    // the value and argument names an expression of generated code reads
    static std::vector<std::string> names_in(const std::string& x) {
        std::vector<std::string> out;
        size_t i = 0;
        auto word = [](char ch) { return std::isalnum(static_cast<unsigned char>(ch)) || ch == '_'; };
        while (i < x.size()) {
            if (!word(x[i])) {
                ++i;
                continue;
            }
            size_t j = i;
            while (j < x.size() && word(x[j])) ++j;
            const std::string id = x.substr(i, j - i);
            const bool after_scope = i >= 2 && x[i - 1] == ':' && x[i - 2] == ':';
            if (!after_scope && !std::isdigit(static_cast<unsigned char>(id[0]))) {
                if (id.size() > 1 && id[0] == 'v' && std::all_of(id.begin() + 1, id.end(), [](char ch) {
                        return std::isdigit(static_cast<unsigned char>(ch));
                    })) {
                    out.push_back(id);
                } else if (id == "h") {
                    out.push_back("h");
                } else if ((id == "sw" || id == "sn") && j < x.size() && x[j] == '[') {
                    const size_t k = x.find(']', j);
                    out.push_back(x.substr(i, k + 1 - i));
                }
            }
            i = j;
        }
        return out;
    }

    int W() const { return W_; }

    std::vector<Node> tape;

private:
    Val reduce(const std::string& op, const std::vector<Val>& pos, const std::map<std::string, Form>& kws);
    int W_;
    bool vector_;
    int next_ = 0;
};

const char* kArith[][2] = {{"+", "__fadd_rn"}, {"-", "__fsub_rn"}, {"*", "__fmul_rn"}, {"/", "__fdiv_rn"}};
const char* kCompare[][2] = {{"<", "<"}, {"<=", "<="}, {">", ">"}, {">=", ">="}, {"=", "=="}, {"!=", "!="}};
const char* kUnary[][2] = {{"exp", "expf"},   {"log", "logf"},   {"tanh", "tanhf"}, {"sin", "sinf"},
                           {"cos", "cosf"},   {"acos", "acosf"}, {"asin", "asinf"}, {"rsqrt", "rsqrtf"},
                           {"abs", "fabsf"},  {"sqrt", "__fsqrt_rn"}};
const char* kBinaryFn[][2] = {{"pow", "powf"},
                              {"atan2", "atan2f"},
                              {"maximum", "es::ieee_maximum"},
                              {"minimum", "es::ieee_minimum"}};

template <size_t N>
const char* lookup(const char* (&table)[N][2], const std::string& key) {
    for (size_t i = 0; i < N; ++i)
        if (key == table[i][0]) return table[i][1];
    return nullptr;
}

// the table's own spelling of an operation (a name that outlives the call)
template <size_t N>
const char* lookup_name(const char* (&table)[N][2], const std::string& key) {
    for (size_t i = 0; i < N; ++i)
        if (key == table[i][0]) return table[i][0];
    return nullptr;
}

double number_arith(const std::string& op, double a, double b) {
    if (op == "+") return a + b;
    if (op == "-") return a - b;
    if (op == "*") return a * b;
    return a / b;
}

bool number_compare(const std::string& op, double a, double b) {
    if (op == "<") return a < b;
    if (op == "<=") return a <= b;
    if (op == ">") return a > b;
    if (op == ">=") return a >= b;
    if (op == "=") return a == b;
    return a != b;
}

Val Tracer::reduce(const std::string& op, const std::vector<Val>& pos, const std::map<std::string, Form>& kws) {
    if (pos.size() != 1) {
        if (op == "max") fail("arity", "(max ...) over tensors takes one value; the elementwise pair is maximum");
        fail("arity", "(sum ...) over tensors takes one value");
    }
    if (!vector_) fail("reduce", "a scalar state's body cannot reduce");
    bool empty_axes = false;
    auto ax = kws.find(":axes");
    if (ax != kws.end()) {
        const Form& a = ax->second;
        if (a.kind != Form::kVec) fail("E-DIM-001", ":axes takes a vector of integers");
        std::vector<long> norm;
        for (const Form& d : a.items) {
            if (d.kind != Form::kNum || d.num != std::floor(d.num)) fail("E-DIM-001", ":axes takes a vector of integers");
            const long n = static_cast<long>(d.num) < 0 ? static_cast<long>(d.num) + 1 : static_cast<long>(d.num);
            if (n != 0) fail("E-DIM-001", "a body value has one axis");
            for (long m : norm)
                if (m == n) fail("E-DIM-001", "an axis is listed twice in :axes");
            norm.push_back(n);
        }
        empty_axes = a.items.empty();
    }
    auto kd = kws.find(":keepdims");
    if (kd != kws.end() && kd->second.kind != Form::kBool) fail("arity", ":keepdims takes true or false");
    Val t = f32(pos[0], "(" + op + " ...)");
    // a one-value vector (or an empty axis list) reduces to itself
    if (empty_axes || !t.wide) return t;
    return emit(false, false, std::string(op == "sum" ? "es::group_sum" : "es::group_max") + "<E, G>(" + t.name +
                                  ", mask)", op == "sum" ? "sum" : "rmax", {t});
}

Val Tracer::eval(const Form& f, const Env& env) {
    switch (f.kind) {
        case Form::kNum: return number(f.num);
        case Form::kBool: return bool_const(f.b);
        case Form::kSym: {
            auto it = env.find(f.s);
            if (it == env.end()) fail("E-SCAN-001", "`" + f.s + "` is not an argument of the body or a let binding");
            return it->second;
        }
        case Form::kKw:
        case Form::kVec: fail("parse", "a keyword or [vector] is not a value here");
        case Form::kList: break;
    }
    if (f.items.empty()) fail("parse", "empty form");
    if (f.items[0].kind != Form::kSym) fail("parse", "a form starts with an operation name");
    const std::string& head = f.items[0].s;
    const std::vector<Form> args(f.items.begin() + 1, f.items.end());

    if (head == "let") {
        if (args.size() < 2 || args[0].kind != Form::kList) fail("arity", "(let ((name value) ...) body)");
        Env inner = env;
        for (const Form& b : args[0].items) {
            if (b.kind != Form::kList || b.items.size() != 2 || b.items[0].kind != Form::kSym)
                fail("arity", "a let binding is (name value)");
            inner[b.items[0].s] = eval(b.items[1], inner);
        }
        Val r;
        for (size_t i = 1; i < args.size(); ++i) r = eval(args[i], inner);
        return r;
    }

    if (head == "sum" || head == "max") {
        std::vector<Val> pos;
        std::map<std::string, Form> kws;
        for (size_t i = 0; i < args.size(); ++i) {
            if (args[i].kind == Form::kKw) {
                if (args[i].s != ":axes" && args[i].s != ":keepdims") fail("arity", "unknown keyword " + args[i].s);
                if (i + 1 >= args.size()) fail("arity", "keyword " + args[i].s + " has no value");
                kws[args[i].s] = args[i + 1];
                ++i;
            } else {
                pos.push_back(eval(args[i], env));
            }
        }
        if (pos.empty()) fail("arity", "(" + head + ") needs a value");
        bool all_numbers = kws.empty();
        for (const Val& v : pos) all_numbers = all_numbers && v.kind == Val::kNumber;
        if (all_numbers) {   // plain numbers: their sum or their maximum
            double r = pos[0].num;
            for (size_t i = 1; i < pos.size(); ++i) r = head == "sum" ? r + pos[i].num : num_max(r, pos[i].num);
            return number(r);
        }
        return reduce(head, pos, kws);
    }

    if (head == "cast") {
        if (args.size() != 2 || args[1].kind != Form::kKw) fail("arity", "(cast x :f32) or (cast x :bool)");
        const Val v = tensor(eval(args[0], env));
        if (args[1].s == ":f32") return v.is_bool ? emit(false, v.wide, "(" + ref(v) + " ? 1.0f : 0.0f)") : v;
        if (args[1].s == ":bool") return v.is_bool ? v : emit(true, v.wide, "(" + ref(v) + " != 0.0f)");
        fail("E-DIM-002", "the body casts only between f32 and bool, not to " + args[1].s);
    }

    if (head == "broadcast-to" || head == "reshape") {
        if (args.size() != 2 || args[1].kind != Form::kVec) fail("arity", "(" + head + " value [dims...])");
        for (const Form& d : args[1].items)
            if (d.kind != Form::kNum) fail("arity", "(" + head + " value [dims...])");
        const Val v = eval(args[0], env);
        if (v.kind != Val::kTensor) return v;
        const auto& dims = args[1].items;
        if (head == "broadcast-to" && !dims.empty() && !v.wide && vector_ && dims.back().num == W_)
            return emit(v.is_bool, true, ref(v), "bcast", {v});
        return v;
    }

    std::vector<Val> vals;
    for (const Form& a : args) vals.push_back(eval(a, env));
    auto arity = [&](size_t lo, long hi) {
        if (vals.size() < lo || (hi >= 0 && vals.size() > static_cast<size_t>(hi)))
            fail("arity", "(" + head + " ...) has a wrong number of arguments: " + std::to_string(vals.size()));
    };

    if (const char* fn = lookup(kArith, head)) {
        arity(1, -1);
        if (vals.size() == 1) {
            const Val& v = vals[0];
            if (v.kind == Val::kNumber) {
                if (head == "-") return number(-v.num);
                if (head == "/") return number(1.0 / v.num);
                return v;
            }
            const Val t = f32(v, head);
            if (head == "-") return emit(false, t.wide, "(-" + ref(t) + ")", "neg", {t});
            if (head == "/") return emit(false, t.wide, "__fdiv_rn(1.0f, " + ref(t) + ")", "div", {tensor(number(1.0)), t});
            return t;
        }
        Val acc = vals[0];
        for (size_t i = 1; i < vals.size(); ++i) {
            const Val& v = vals[i];
            if (acc.kind == Val::kNumber && v.kind == Val::kNumber) {
                acc = number(number_arith(head, acc.num, v.num));
            } else {
                const Val a = f32(acc, head), b = f32(v, head);
                const char* nm = head == "+" ? "add" : head == "-" ? "sub" : head == "*" ? "mul" : "div";
                acc = emit(false, a.wide || b.wide, std::string(fn) + "(" + ref(a) + ", " + ref(b) + ")", nm, {a, b});
            }
        }
        return acc;
    }
    if (const char* op = lookup(kCompare, head)) {
        arity(2, 2);
        if (vals[0].kind == Val::kNumber && vals[1].kind == Val::kNumber)
            return bool_const(number_compare(head, vals[0].num, vals[1].num));
        const Val a = f32(vals[0], head), b = f32(vals[1], head);
        return emit(true, a.wide || b.wide, "(" + ref(a) + " " + op + " " + ref(b) + ")");
    }
    if (head == "and" || head == "or") {
        arity(1, -1);
        Val acc = boolean(vals[0], head);
        for (size_t i = 1; i < vals.size(); ++i) {
            const Val b = boolean(vals[i], head);
            acc = emit(true, acc.wide || b.wide, "(" + ref(acc) + (head == "and" ? " && " : " || ") + ref(b) + ")");
        }
        return acc;
    }
    if (head == "not") {
        arity(1, 1);
        const Val a = boolean(vals[0], "not");
        return emit(true, a.wide, "(!" + ref(a) + ")");
    }
    if (head == "where") {
        arity(3, 3);
        const Val m = boolean(vals[0], "where mask");
        const Val a = tensor(vals[1]), b = tensor(vals[2]);
        if (a.is_bool != b.is_bool) fail("E-DIM-002", "where: branches of different dtypes");
        return emit(a.is_bool, m.wide || a.wide || b.wide, "(" + ref(m) + " ? " + ref(a) + " : " + ref(b) + ")",
                    "where", {a, b}, m);
    }
    if (head == "neg") {
        arity(1, 1);
        const Val a = f32(vals[0], head);
        return emit(false, a.wide, "(-" + ref(a) + ")", "neg", {a});
    }
    if (const char* fn = lookup(kUnary, head)) {
        arity(1, 1);
        // sqrt, exp and log are overloaded: on a plain number they stay plain
        if (vals[0].kind == Val::kNumber && (head == "sqrt" || head == "exp" || head == "log")) {
            const double x = vals[0].num;
            return number(head == "sqrt" ? std::sqrt(x) : head == "exp" ? std::exp(x) : std::log(x));
        }
        const Val a = f32(vals[0], head);
        return emit(false, a.wide, std::string(fn) + "(" + ref(a) + ")", lookup_name(kUnary, head), {a});
    }
    if (const char* fn = lookup(kBinaryFn, head)) {
        arity(2, 2);
        if (head == "pow" && vals[0].kind == Val::kNumber && vals[1].kind == Val::kNumber)
            return number(std::pow(vals[0].num, vals[1].num));
        const Val a = f32(vals[0], head), b = f32(vals[1], head);
        return emit(false, a.wide || b.wide, std::string(fn) + "(" + ref(a) + ", " + ref(b) + ")",
                    lookup_name(kBinaryFn, head), {a, b});
    }
    fail("op", "`" + head + "` is not an operation a body may use");
}

// ---------------------------------------------------------------------------
// the vector-Jacobian product: the tape swept backwards
//
// Derivatives ("Precision and gradients": comparisons and casts have none,
// `where` follows the selected branch, the usual tie rules apply), each an
// f32 expression rounded step by step:
//   a+b: (g, g)   a-b: (g, -g)   a*b: (g*b, g*a)   a/b: (g/b, -(g*q)/b), q = a/b
//   -a: -g   |a|: g*sign(a) (0 at 0)   sqrt: (g*0.5)/out   exp: g*out
//   log: g/a   tanh: g*(1-out*out)   sin: g*cos(a)   cos: -(g*sin(a))
//   rsqrt: g*((out*out*out)*-0.5)   acos: -(g/sqrt(1-a*a))   asin: g/sqrt(1-a*a)
//   atan2(y, x): ((g*x)/(x*x+y*y), -(g*y)/(x*x+y*y))
//   pow(a, b): (g*(b*pow(a, b-1)), 0 if out == 0 else g*(out*log(a)))
//   maximum / minimum: the larger (smaller) operand takes g, a tie or NaN
//   splits g*0.5 each; where: g to the selected branch; sum: g to every
//   value; max: g/count to each of its count equal maxima.
// Contributions reach an operand in reverse tape order, a node's operands in
// argument order, the first assigned and later ones added; a width-one
// operand of a wide operation receives the sum of the wide contribution over
// the state (this thread's values in order, then the lane's threads).
class Adjoint {
public:
    // `result`: the body's value; when `from_saved` its derivative formulas
    // read the trip's output from the saved states (`res`), which hold it
    Adjoint(const Tracer& tr, const Val& result, bool from_saved)
        : tr_(tr), res_name_(result.name), from_saved_(from_saved) {}

    std::string code;
    std::set<std::string> used;     // forward values the derivatives read
    bool reads_res = false;

    // a forward value as a derivative formula reads it
    std::string val(const Val& x) {
        if (x.kind == Val::kTensor && from_saved_ && x.name == res_name_) {
            reads_res = true;
            return "res[e]";
        }
        if (x.kind == Val::kTensor) used.insert(x.name);
        return tr_.ref(x);
    }

    static std::string gname(const Val& v) {
        std::string g = "g_";
        for (char ch : v.name)
            if (ch != '[' && ch != ']') g += ch;
        return g;
    }

    bool has(const Val& v) const { return assigned_.count(gname(v)) != 0; }

    // the seed: the cotangent of the body's result is the state's cotangent
    // (a width-one result, spread over the state, takes its sum)
    void seed(const Val& r) {
        if (r.kind != Val::kTensor || !r.diff) return;
        contribute(r, "lam[e]", true);
    }

    void sweep() {
        const std::vector<Node>& tape = tr_.tape;
        for (auto it = tape.rbegin(); it != tape.rend(); ++it) {
            const Node& n = *it;
            if (!has(n.out)) continue;
            const bool w = n.out.wide;
            const std::string G = w ? gname(n.out) + "[e]" : gname(n.out);
            const Val& a = n.args[0];
            const Val* b = n.args.size() > 1 ? &n.args[1] : nullptr;
            const std::string& op = n.op;
            // the operands' and the result's values, only where a formula reads them
            static const std::set<std::string> kReadsA = {"mul", "abs", "log", "sin", "cos", "acos", "asin",
                                                          "atan2", "pow", "maximum", "minimum", "rmax"};
            static const std::set<std::string> kReadsB = {"mul", "div", "atan2", "pow", "maximum", "minimum"};
            static const std::set<std::string> kReadsOut = {"div", "sqrt", "exp", "tanh", "rsqrt", "pow", "rmax"};
            const std::string A = kReadsA.count(op) ? val(a) : "";
            const std::string B = b && kReadsB.count(op) ? val(*b) : "";
            const std::string OUT = kReadsOut.count(op) ? val(n.out) : "";
            auto half = "__fmul_rn(" + G + ", 0.5f)";
            if (op == "add") {
                contribute(a, G, w);
                contribute(*b, G, w);
            } else if (op == "sub") {
                contribute(a, G, w);
                contribute(*b, "(-" + G + ")", w);
            } else if (op == "mul") {
                contribute(a, "__fmul_rn(" + G + ", " + B + ")", w);
                contribute(*b, "__fmul_rn(" + G + ", " + A + ")", w);
            } else if (op == "div") {
                contribute(a, "__fdiv_rn(" + G + ", " + B + ")", w);
                contribute(*b, "(-__fdiv_rn(__fmul_rn(" + G + ", " + OUT + "), " + B + "))", w);
            } else if (op == "neg") {
                contribute(a, "(-" + G + ")", w);
            } else if (op == "abs") {
                contribute(a, "(" + A + " > 0.0f ? " + G + " : (" + A + " < 0.0f ? (-" + G + ") : 0.0f))", w);
            } else if (op == "sqrt") {
                contribute(a, "__fdiv_rn(" + half + ", " + OUT + ")", w);
            } else if (op == "exp") {
                contribute(a, "__fmul_rn(" + G + ", " + OUT + ")", w);
            } else if (op == "log") {
                contribute(a, "__fdiv_rn(" + G + ", " + A + ")", w);
            } else if (op == "tanh") {
                contribute(a, "__fmul_rn(" + G + ", __fsub_rn(1.0f, __fmul_rn(" + OUT + ", " + OUT + ")))", w);
            } else if (op == "sin") {
                contribute(a, "__fmul_rn(" + G + ", cosf(" + A + "))", w);
            } else if (op == "cos") {
                contribute(a, "(-__fmul_rn(" + G + ", sinf(" + A + ")))", w);
            } else if (op == "rsqrt") {
                contribute(a, "__fmul_rn(" + G + ", __fmul_rn(__fmul_rn(__fmul_rn(" + OUT + ", " + OUT + "), " + OUT +
                                  "), -0.5f))", w);
            } else if (op == "acos" || op == "asin") {
                const std::string q = "__fdiv_rn(" + G + ", __fsqrt_rn(__fsub_rn(1.0f, __fmul_rn(" + A + ", " + A + "))))";
                contribute(a, op == "acos" ? "(-" + q + ")" : q, w);
            } else if (op == "atan2") {
                const std::string den = "__fadd_rn(__fmul_rn(" + B + ", " + B + "), __fmul_rn(" + A + ", " + A + "))";
                contribute(a, "__fdiv_rn(__fmul_rn(" + G + ", " + B + "), " + den + ")", w);
                contribute(*b, "(-__fdiv_rn(__fmul_rn(" + G + ", " + A + "), " + den + "))", w);
            } else if (op == "pow") {
                contribute(a, "__fmul_rn(" + G + ", __fmul_rn(" + B + ", powf(" + A + ", __fsub_rn(" + B + ", 1.0f))))", w);
                contribute(*b, "(" + OUT + " == 0.0f ? 0.0f : __fmul_rn(" + G + ", __fmul_rn(" + OUT + ", logf(" + A +
                                   "))))", w);
            } else if (op == "maximum" || op == "minimum") {
                const char* cmp = op == "maximum" ? " > " : " < ";
                contribute(a, "(" + A + cmp + B + " ? " + G + " : (" + B + cmp + A + " ? 0.0f : " + half + "))", w);
                contribute(*b, "(" + B + cmp + A + " ? " + G + " : (" + A + cmp + B + " ? 0.0f : " + half + "))", w);
            } else if (op == "where") {
                const std::string M = val(n.mask);
                contribute(a, "(" + M + " ? " + G + " : 0.0f)", w);
                contribute(*b, "(" + M + " ? 0.0f : " + G + ")", w);
            } else if (op == "sum") {
                contribute(a, G, true);     // every value of the reduced vector
            } else if (op == "rmax") {
                const std::string cnt = "cnt" + std::to_string(tmp_++);
                code += "        float " + cnt + "_v[E];\n#pragma unroll\n        for (int e = 0; e < E; ++e) " + cnt +
                        "_v[e] = (" + A + " == " + OUT + ") ? 1.0f : 0.0f;\n        const float " + cnt +
                        " = es::group_sum<E, G>(" + cnt + "_v, mask);\n";
                contribute(a, "(" + A + " == " + OUT + " ? __fdiv_rn(" + G + ", " + cnt + ") : 0.0f)", true);
            } else if (op == "bcast") {
                contribute(a, G, true);
            }
        }
    }

    // the forward statements the derivatives need: the values they read and
    // everything those are computed from, in the trace's order
    std::string live_forward(std::set<std::string>* live) const {
        std::map<std::string, const Tracer::Stmt*> def;
        for (const Tracer::Stmt& st : tr_.stmts) def[st.name] = &st;
        std::vector<std::string> todo(used.begin(), used.end());
        while (!todo.empty()) {
            const std::string nm = todo.back();
            todo.pop_back();
            if (!live->insert(nm).second) continue;
            auto it = def.find(nm);
            if (it != def.end())
                for (const std::string& d : it->second->deps) todo.push_back(d);
        }
        std::string out;
        for (const Tracer::Stmt& st : tr_.stmts)
            if (live->count(st.name)) out += st.code;
        return out;
    }

    // the gradient of a leaf, or zero
    std::string grad_or_zero(const Val& v) const {
        if (!has(v)) return "0.0f";
        return v.wide ? gname(v) + "[e]" : gname(v);
    }

private:
    // add `expr` (wide: an expression of e) to the gradient of `target`
    void contribute(const Val& target, const std::string& expr, bool expr_wide) {
        if (target.kind != Val::kTensor || !target.diff) return;
        const std::string gv = gname(target);
        std::string value = expr;
        bool value_wide = expr_wide;
        if (expr_wide && !target.wide) {
            // a width-one operand of a wide operation: the sum over the state
            const std::string c = "c" + std::to_string(tmp_++);
            code += "        float " + c + "[E];\n#pragma unroll\n        for (int e = 0; e < E; ++e) " + c + "[e] = " +
                    expr + ";\n        const float " + c + "_s = es::group_sum<E, G>(" + c + ", mask);\n";
            value = c + "_s";
            value_wide = false;
        }
        const bool first = assigned_.insert(gv).second;
        if (target.wide) {
            // a wide target takes a wide value, or a width-one one on every value
            const std::string rhs = first ? value : "__fadd_rn(" + gv + "[e], " + value + ")";
            if (first) code += "        float " + gv + "[E];\n";
            code += "#pragma unroll\n        for (int e = 0; e < E; ++e) " + gv + "[e] = " + rhs + ";\n";
        } else {
            (void)value_wide;
            if (first) code += "        float " + gv + " = " + value + ";\n";
            else code += "        " + gv + " = __fadd_rn(" + gv + ", " + value + ");\n";
        }
    }

    const Tracer& tr_;
    std::string res_name_;
    bool from_saved_;
    std::set<std::string> assigned_;
    int tmp_ = 0;
};

std::string comment_safe(const std::string& s) {
    std::string r;
    for (size_t i = 0; i < s.size(); ++i) {
        if (s[i] == '*' && i + 1 < s.size() && s[i + 1] == '/') {
            r += "* /";
            ++i;
        } else {
            r += s[i];
        }
    }
    return r;
}

}  // namespace

std::unique_ptr<Program> Program::parse(const std::string& text) {
    Form f = Reader(text).read_all();
    if (f.kind != Form::kList || f.items.size() < 3 || f.items[0].kind != Form::kSym || f.items[0].s != "lambda" ||
        f.items[1].kind != Form::kList)
        fail("parse", "a body is (lambda (h seq ...) expr)");
    std::unique_ptr<Program> p(new Program());
    p->text_ = text;
    for (const Form& a : f.items[1].items) {
        if (a.kind != Form::kSym) fail("arity", "the body's arguments are names");
        for (const std::string& q : p->params_)
            if (q == a.s) fail("arity", "repeated argument name `" + a.s + "`");
        p->params_.push_back(a.s);
    }
    if (p->params_.size() < 2) fail("arity", "a body takes the state and at least one sequence");
    p->exprs_.assign(f.items.begin() + 2, f.items.end());
    return p;
}

std::string Program::generate(int W, bool vector, unsigned wide_mask, bool with_vjp) const {
    const int ns = n_seqs();
    Tracer tr(W, vector);
    Env env;
    Val h;
    h.kind = Val::kTensor;
    h.name = "h";
    h.wide = true;
    h.diff = true;
    env[params_[0]] = h;
    int nw = 0, nn = 0;
    std::vector<Val> leaves;
    for (int k = 0; k < ns; ++k) {
        Val s;
        s.kind = Val::kTensor;
        s.wide = (wide_mask >> k) & 1u;
        s.diff = true;
        s.name = s.wide ? "sw[" + std::to_string(nw++) + "]" : "sn[" + std::to_string(nn++) + "]";
        env[params_[k + 1]] = s;
        leaves.push_back(s);
    }
    Val r;
    for (const Form& e : exprs_) r = tr.eval(e, env);
    if (r.kind == Val::kBoolConst || (r.kind == Val::kTensor && r.is_bool))
        fail("E-DIM-002", "the body returns bool; it must return f32");
    r = tr.tensor(r);
    if (!r.wide && W != 1)
        fail("E-DIM-001", "the body returns one value; the state has width " + std::to_string(W));

    std::ostringstream o;
    o << "// functor for the body\n";
    std::istringstream lines(comment_safe(text_));
    for (std::string line; std::getline(lines, line);) o << "//   " << line << "\n";
    o << "// state width " << W
      << (vector ? " (vector state)" : " (scalar state)") << ", " << ns << " sequence(s), wide mask 0x" << std::hex
      << wide_mask << std::dec << "\n";
    o << "struct EsBody {\n";
    o << "    static constexpr int kNS = " << ns << ";\n";
    o << "    static constexpr unsigned kWideMask = 0x" << std::hex << wide_mask << std::dec << "u;\n";
    o << "    static constexpr int kSW = " << (nw > 0 ? nw : 1) << ";\n";
    o << "    static constexpr int kSN = " << (nn > 0 ? nn : 1) << ";\n";
    o << "    template <int E, int G>\n";
    o << "    __device__ __forceinline__ static void step(float (&r)[E], const float (&h)[E],\n"
         "                                                const float (&sw)[kSW][E], const float (&sn)[kSN],\n"
         "                                                const unsigned mask) {\n";
    o << "        (void)h;\n        (void)sw;\n        (void)sn;\n        (void)mask;\n";
    o << tr.code;
    o << "#pragma unroll\n        for (int e = 0; e < E; ++e) r[e] = " << tr.ref(r) << ";\n";
    o << "    }\n";
    if (with_vjp) {
        // the trip's vector-Jacobian product: the body again from the state
        // before the trip (`h`), then the tape backwards from the cotangent
        // `lam` of the state after it (`res`); dp is the previous state's
        // cotangent, dsw / dsn the sequences' (a width-one one summed over
        // the state)
        // The trip's result is read from the saved states (they hold it);
        // the other values the derivatives read are computed again, and only
        // those.  A sequence no needed value reads is not needed at all.
        const bool computed_result = r.kind == Val::kTensor && r.wide && r.name.size() > 1 && r.name[0] == 'v';
        Adjoint adj(tr, r, computed_result);
        adj.seed(r);
        adj.sweep();
        std::set<std::string> live;
        const std::string forward = adj.live_forward(&live);
        unsigned seq_mask = 0;
        {
            int kw = 0, kn = 0;
            for (int k = 0; k < ns; ++k) {
                const bool wide = (wide_mask >> k) & 1u;
                const std::string nm = wide ? "sw[" + std::to_string(kw++) + "]" : "sn[" + std::to_string(kn++) + "]";
                if (live.count(nm)) seq_mask |= 1u << k;
            }
        }
        o << "    // sequences the vector-Jacobian product reads (bit k), and whether it\n"
             "    // reads the trip's result from the saved states\n";
        o << "    static constexpr unsigned kVjpSeqs = 0x" << std::hex << seq_mask << std::dec << "u;\n";
        o << "    static constexpr bool kVjpRes = " << (adj.reads_res ? "true" : "false") << ";\n";
        o << "    template <int E, int G>\n";
        o << "    __device__ __forceinline__ static void vjp(float (&dp)[E], float (&dsw)[kSW][E], float (&dsn)[kSN],\n"
             "                                               const float (&lam)[E], const float (&h)[E],\n"
             "                                               const float (&res)[E],\n"
             "                                               const float (&sw)[kSW][E], const float (&sn)[kSN],\n"
             "                                               const unsigned mask) {\n";
        o << "        (void)lam;\n        (void)h;\n        (void)res;\n        (void)sw;\n        (void)sn;\n"
             "        (void)mask;\n";
        o << forward << adj.code;
        o << "#pragma unroll\n        for (int e = 0; e < E; ++e) dp[e] = " << adj.grad_or_zero(h) << ";\n";
        int qw = 0, qn = 0;
        for (const Val& s : leaves) {
            if (s.wide)
                o << "#pragma unroll\n        for (int e = 0; e < E; ++e) dsw[" << qw++ << "][e] = " << adj.grad_or_zero(s)
                  << ";\n";
            else
                o << "        dsn[" << qn++ << "] = " << adj.grad_or_zero(s) << ";\n";
        }
        if (nw == 0) o << "#pragma unroll\n        for (int e = 0; e < E; ++e) dsw[0][e] = 0.0f;\n";
        if (nn == 0) o << "        dsn[0] = 0.0f;\n";
        o << "    }\n";
    }
    o << "};\n";
    return o.str();
}

}  // namespace body
}  // namespace es
