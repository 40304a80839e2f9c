// es_body_compiler.h -- body programs: reading, checking and translating an
// element-scan body given as text into a CUDA functor for the kernel
// skeletons (skel_common.cuh describes the functor).  Host code only.
#pragma once

#include <memory>
#include <string>
#include <vector>

namespace es {
namespace body {

// A body the contract rejects.  `code` classifies it: "parse", "arity",
// "E-SCAN-001" (a name that is no argument or binding), "reduce" (a scalar
// state's body reduces), "op" (not a body operation), "E-DIM-001" (widths,
// axes), "E-DIM-002" (f32 / bool mismatch).
struct Error {
    std::string code;
    std::string msg;
};

// One read s-expression: a number, `true`/`false`, a symbol, a :keyword, a
// [vector] or a (list).
struct Form {
    enum Kind { kNum, kBool, kSym, kKw, kVec, kList } kind = kNum;
    double num = 0.0;
    bool b = false;
    std::string s;
    std::vector<Form> items;
};

// A parsed (lambda (h seq ...) expr ...).
class Program {
public:
    int n_seqs() const { return static_cast<int>(params_.size()) - 1; }
    const std::string& text() const { return text_; }

    // The functor for one call signature: state width W (1 for a scalar
    // state), whether the state is a vector (`:state-axis`), and which
    // sequences are as wide as the state (bit k of wide_mask).  With
    // `with_vjp` it also has the trip's vector-Jacobian product.  Throws Error.
    std::string generate(int W, bool vector, unsigned wide_mask, bool with_vjp = false) const;

    // Throws Error when the text is not a body.
    static std::unique_ptr<Program> parse(const std::string& text);

private:
    Program() = default;
    std::string text_;
    std::vector<std::string> params_;
    std::vector<Form> exprs_;
};

}  // namespace body
}  // namespace es
