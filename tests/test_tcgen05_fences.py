"""tcgen05 fence lint over the CUDA sources (CPU only).

The page "[None][feat] Share Kimi K3 FP4 modeling and add NVFP4 support on
SM103" (NVIDIA/TensorRT-LLM PR #20532) holds its tcgen05 kernels to a fence
rule that a test reads out of their sources (the commit extending
test_k3_tcgen05_fences.py to the weight-stream kernels).  Restated:

  A. a tcgen05 operation (MMA, commit, TMEM load/store, alloc/dealloc) that a
     thread reaches after waiting on another thread (an mbarrier wait, a CTA
     or named barrier) must be preceded, after that wait, by
     tcgen05.fence::after_thread_sync;
  B. an arrive or a barrier that a thread reaches after touching tensor
     memory (a TMEM load or store, or the wait for one) must be preceded,
     after that access, by tcgen05.fence::before_thread_sync.

The lint parses every __global__ function of csrc/*.cu into its statements,
if/else branches, loops and lambdas, and runs a may-analysis over every path
(branches join, loop bodies are iterated to a fixed point, a lambda's body is
analysed where it is called).  Mutants remove single fences from the real
kernel source and must be caught."""
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CSRC = os.path.join(ROOT, "speculative_decoding_drafter_k3_gb300", "csrc")

# ------------------------------------------------------------ preprocessing --


def _strip(src):
    """Comments and preprocessor lines become blanks (newlines kept, so
    offsets keep their line numbers); every string or character literal
    becomes "@<k>" with its contents in the returned table."""
    out, strings, i, n = [], [], 0, len(src)
    at_line_start = True
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            j = n if j < 0 else j
            out.append(" " * (j - i))
            i = j
            continue
        if src.startswith("/*", i):
            j = src.find("*/", i + 2)
            j = n if j < 0 else j + 2
            out.append(re.sub(r"[^\n]", " ", src[i:j]))
            i = j
            continue
        if at_line_start and c == "#":
            j = src.find("\n", i)
            j = n if j < 0 else j
            out.append(" " * (j - i))
            i = j
            continue
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            strings.append(src[i + 1:j])
            tag = f'"@{len(strings) - 1}"'
            body = src[i:j + 1]
            # Keep the literal's newlines so later line numbers stay right.
            out.append(tag + "\n" * body.count("\n") + " " * max(0, len(body) - len(tag) - body.count("\n")))
            i = j + 1
            at_line_start = False
            continue
        out.append(c)
        if c == "\n":
            at_line_start = True
        elif not c.isspace():
            at_line_start = False
        i += 1
    return "".join(out), strings


# ------------------------------------------------------------------ parser --

class Stmt:
    def __init__(self, text, pos):
        self.text, self.pos = text, pos


class Block:
    def __init__(self, items):
        self.items = items


class If:
    def __init__(self, cond, then, other):
        self.cond, self.then, self.other = cond, then, other


class Loop:
    def __init__(self, head, body):
        self.head, self.body = head, body


_OPEN, _CLOSE = "([{", ")]}"
_LAMBDA = re.compile(r"\bauto\s+(\w+)\s*=\s*\[[^\]]*\]\s*(\([^)]*\))?\s*(->\s*[\w:<>\s*&]+)?\s*\{")


class Parser:
    def __init__(self, text, base=0):
        self.t, self.i, self.base = text, 0, base
        self.lambdas = {}

    def ws(self):
        while self.i < len(self.t) and self.t[self.i].isspace():
            self.i += 1

    def word(self):
        m = re.match(r"[A-Za-z_]\w*", self.t[self.i:])
        return m.group(0) if m else None

    def match(self, i):
        """Index just past the bracket group opening at i."""
        depth = 0
        for j in range(i, len(self.t)):
            if self.t[j] in _OPEN:
                depth += 1
            elif self.t[j] in _CLOSE:
                depth -= 1
                if depth == 0:
                    return j + 1
        raise ValueError("unbalanced brackets")

    def group(self):
        self.ws()
        assert self.t[self.i] == "(", self.t[self.i:self.i + 40]
        j = self.match(self.i)
        g = Stmt(self.t[self.i:j], self.base + self.i)
        self.i = j
        return g

    def block_items(self):
        items = []
        while True:
            self.ws()
            if self.i >= len(self.t) or self.t[self.i] == "}":
                return items
            items.append(self.stmt())

    def stmt(self):
        self.ws()
        if self.t[self.i] == "{":
            self.i += 1
            items = self.block_items()
            assert self.t[self.i] == "}"
            self.i += 1
            return Block(items)
        w = self.word()
        if w == "if":
            self.i += 2
            self.ws()
            if self.word() == "constexpr":
                self.i += len("constexpr")
            cond = self.group()
            then = self.stmt()
            self.ws()
            other = None
            if self.word() == "else":
                self.i += 4
                other = self.stmt()
            return If(cond, then, other)
        if w in ("for", "while"):
            self.i += len(w)
            head = self.group()
            return Loop(head, self.stmt())
        if w == "do":
            self.i += 2
            body = self.stmt()
            self.ws()
            assert self.word() == "while"
            self.i += 5
            head = self.group()
            self.ws()
            assert self.t[self.i] == ";"
            self.i += 1
            return Block([body, Loop(head, body)])
        # A plain statement, up to its ';' outside any bracket.
        start, depth, j = self.i, 0, self.i
        while True:
            c = self.t[j]
            if c in _OPEN:
                depth += 1
            elif c in _CLOSE:
                depth -= 1
            elif c == ";" and depth == 0:
                break
            j += 1
        text = self.t[start:j]
        self.i = j + 1
        m = _LAMBDA.search(text)
        if m:
            # A lambda definition: its body runs where the lambda is called.
            b0 = start + m.end() - 1
            b1 = self.match(b0)
            sub = Parser(self.t[b0 + 1:b1 - 1], self.base + b0 + 1)
            sub.lambdas = self.lambdas
            self.lambdas[m.group(1)] = Block(sub.block_items())
            return Stmt(text[:m.start()], self.base + start)
        return Stmt(text, self.base + start)


# ---------------------------------------------------------------- analysis --

WAITS = ("mbar_wait", "mbar_wait_slow", "mbar_try_wait")
BARRIERS = ("named_bar_sync", "__syncthreads")
SIGNALS = ("mbar_arrive", "mbar_arrive_expect_tx", "__syncwarp")
TC_CALLS = ("mma_ss", "mma_ts", "mma_commit", "tmem_ld_h32", "tmem_ld_h16", "tmem_st_h32", "tmem_st_h16",
            "tmem_st32")
TMEM_TOUCH = ("tmem_ld_h32", "tmem_ld_h16", "tmem_st_h32", "tmem_st_h16", "tmem_st32", "tmem_wait_st")
_CALL = re.compile(r"\b([A-Za-z_]\w*)\s*\(")
_STR = re.compile(r'"@(\d+)"')


def events(text, strings, lambdas):
    """(offset, kind, name) of every event in a plain statement, in order."""
    evs = []
    for m in _CALL.finditer(text):
        name = m.group(1)
        kinds = []
        if name == "fence_after":
            kinds.append("fence_after")
        if name == "fence_before":
            kinds.append("fence_before")
        if name in WAITS:
            kinds.append("wait")
        if name in BARRIERS:
            kinds += ["signal", "wait"]
        if name in SIGNALS:
            kinds.append("signal")
        if name in TC_CALLS:
            kinds.append("tc_op")
        if name in TMEM_TOUCH:
            kinds.append("tmem")
        if name in lambdas:
            kinds.append("call")
        for k in kinds:
            evs.append((m.start(), k, name))
    for m in _STR.finditer(text):
        s = strings[int(m.group(1))]
        if "tcgen05.fence::after_thread_sync" in s:
            evs.append((m.start(), "fence_after", "asm"))
        elif "tcgen05.fence::before_thread_sync" in s:
            evs.append((m.start(), "fence_before", "asm"))
        elif re.search(r"tcgen05\.wait::(ld|st)", s):
            evs.append((m.start(), "tmem", "asm wait"))
        elif re.search(r"tcgen05\.(mma|commit|ld|st|alloc|dealloc|relinquish|cp|shift)", s):
            evs.append((m.start(), "tc_op", s.split()[0]))
            if re.search(r"tcgen05\.(ld|st)", s):
                evs.append((m.start() + 1, "tmem", s.split()[0]))
        if re.search(r"\bmbarrier\.(try_wait|test_wait)", s):
            evs.append((m.start(), "wait", "asm mbarrier wait"))
        if re.search(r"\bmbarrier\.arrive", s) or re.search(r"\bbar(rier)?\.(sync|arrive)", s):
            evs.append((m.start(), "signal", "asm arrive/barrier"))
    return sorted(evs)


class Lint:
    """State: (a, b) = (witness of a wait not yet followed by fence_after,
    witness of a TMEM access not yet followed by fence_before), or None."""

    def __init__(self, fname, text, strings, line_of):
        self.fname, self.text, self.strings, self.line_of = fname, text, strings, line_of
        self.found = set()

    def join(self, s1, s2):
        return (s1[0] or s2[0], s1[1] or s2[1])

    def apply(self, stmt, st, lambdas, depth=0):
        a, b = st
        for off, kind, name in events(stmt.text, self.strings, lambdas):
            line = self.line_of(stmt.pos + off)
            if kind == "fence_after":
                a = None
            elif kind == "fence_before":
                b = None
            elif kind == "signal":
                if b is not None:
                    self.found.add((self.fname, line, "B", f"{name} after a TMEM access at line {b} "
                                                           f"without tcgen05.fence::before_thread_sync"))
            elif kind == "wait":
                a = line
            elif kind == "tc_op":
                if a is not None:
                    self.found.add((self.fname, line, "A", f"{name} after a wait at line {a} "
                                                           f"without tcgen05.fence::after_thread_sync"))
            elif kind == "tmem":
                b = line
            elif kind == "call" and depth < 8:
                a, b = self.run(lambdas[name], (a, b), lambdas, depth + 1)
        return (a, b)

    def run(self, node, st, lambdas, depth=0):
        if node is None:
            return st
        if isinstance(node, Stmt):
            return self.apply(node, st, lambdas, depth)
        if isinstance(node, Block):
            for n in node.items:
                st = self.run(n, st, lambdas, depth)
            return st
        if isinstance(node, If):
            st = self.apply(node.cond, st, lambdas, depth)
            return self.join(self.run(node.then, st, lambdas, depth), self.run(node.other, st, lambdas, depth))
        if isinstance(node, Loop):
            head = self.apply(node.head, st, lambdas, depth)
            for _ in range(8):
                end = self.run(node.body, head, lambdas, depth)
                nxt = self.join(head, self.apply(node.head, end, lambdas, depth))
                if (nxt[0] is None) == (head[0] is None) and (nxt[1] is None) == (head[1] is None):
                    return nxt
                head = nxt
            return head
        raise TypeError(node)


def lint_source(src, fname="<src>"):
    """Fence-rule violations of every __global__ function in `src`:
    a sorted list of (file, line, rule, message)."""
    text, strings = _strip(src)
    starts = [0] + [m.end() for m in re.finditer("\n", text)]

    def line_of(off):
        lo, hi = 0, len(starts) - 1
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if starts[mid] <= off:
                lo = mid
            else:
                hi = mid - 1
        return lo + 1

    lint = Lint(fname, text, strings, line_of)
    for m in re.finditer(r"__global__\b", text):
        p = Parser(text)
        # The body is the first brace outside the signature's parentheses.
        depth, b0 = 0, m.end()
        while not (text[b0] == "{" and depth == 0):
            depth += text[b0] == "("
            depth -= text[b0] == ")"
            b0 += 1
        b1 = p.match(b0)
        body = Parser(text[b0 + 1:b1 - 1], b0 + 1)
        items = body.block_items()
        lint.run(Block(items), (None, None), body.lambdas)
    return sorted(lint.found)


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith((".cu", ".cuh")))


def tc_kernel_source():
    return open(os.path.join(CSRC, "k3da.cu")).read()


# ------------------------------------------------------------------- tests --

def test_every_kernel_source_follows_the_fence_rule():
    found = []
    for path in sources():
        found += lint_source(open(path).read(), os.path.basename(path))
    assert not found, "\n".join(f"{f}:{ln}: rule {r}: {msg}" for f, ln, r, msg in found)


def test_the_lint_reads_the_tcgen05_kernel():
    """The kernel source really holds the operations the rule is about."""
    text, _ = _strip(tc_kernel_source())
    for name in ("mma_ss(", "mma_ts(", "mma_commit(", "tmem_ld_h32(", "tmem_st_h16(", "fence_after()",
                 "fence_before()", "mbar_wait(", "mbar_arrive("):
        assert name in text, name


def _remove(src, anchor, fence, after=True):
    """src with the first `fence` after (or before) the first `anchor` removed."""
    i = src.index(anchor)
    if after:
        j = src.index(fence, i)
    else:
        j = src.rindex(fence, 0, i)
    return src[:j] + src[j + len(fence):]


MUTANTS = {
    # the wait for S of an item, then its TMEM load
    "no_fence_after_s_full_wait": ("mbar_wait(bar_sfull + 8 * b", "fence_after();", True, "A"),
    # the wait for P of an item, then the P.V MMA
    "no_fence_after_p_full_wait": ("mbar_wait(bar_pfull + 8 * b, ph", "fence_after();", True, "A"),
    # the P.V that freed an S/P buffer, then the next QK^T into it
    "no_fence_after_buffer_free_wait": ("mbar_wait(bar_odone + 8 * b, ph ^ 1u", "fence_after();", True, "A"),
    # the page's TMA data, then the QK^T MMA
    "no_fence_after_page_wait": ("mbar_wait(bar_full + 8 * s, static_cast<uint32_t>(((kr - 1) / kStages) & 1)",
                                 "fence_after();", True, "A"),
    # P stored to TMEM, then the arrive that hands it to the P.V warp
    "no_fence_before_p_handover": ("mbar_arrive(bar_pfull + 8 * b)", "fence_before();", False, "B"),
    # the final CTA barrier, then the TMEM dealloc
    "no_fence_after_final_barrier": ("tcgen05.dealloc", "fence_after();", False, "A"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_the_lint_catches_a_removed_fence(name):
    anchor, fence, after, rule = MUTANTS[name]
    src = tc_kernel_source()
    assert not lint_source(src)
    bad = lint_source(_remove(src, anchor, fence, after))
    assert any(r == rule for _, _, r, _ in bad), name


@pytest.mark.parametrize("body,rules", [
    # a fence on one branch only leaves the other path unfenced
    ("mbar_wait(x, 0); if (c) { fence_after(); } mma_ss(d, a, b, i, 0);", {"A"}),
    ("mbar_wait(x, 0); fence_after(); if (c) { mma_ss(d, a, b, i, 0); }", set()),
    ("if (c) { mbar_wait(x, 0); fence_after(); } else { mbar_wait(y, 0); } tmem_st32(t, r);", {"A"}),
    # the loop's back edge carries the wait at the end of the body
    ("for (;;) { tmem_ld_h32(t, r); fence_before(); mbar_wait(x, 0); }", {"A"}),
    ("for (;;) { mbar_wait(x, 0); fence_after(); tmem_ld_h32(t, r); fence_before(); }", set()),
    ("while (!mbar_try_wait(x, 0)) {} mma_commit(x);", {"A"}),
    # a lambda's body counts where it is called
    ("auto f = [&]() { tmem_ld_h32(t, r); }; mbar_wait(x, 0); f();", {"A"}),
    ("auto f = [&]() { tmem_ld_h32(t, r); }; mbar_wait(x, 0); fence_after(); f(); fence_before();", set()),
    # rule B: a TMEM access before an arrive or a barrier
    ("tmem_ld_h32(t, r); mbar_arrive(x);", {"B"}),
    ("tmem_st_h16(t, r); tmem_wait_st(); fence_before(); __syncwarp(); mbar_arrive(x);", set()),
    ("tmem_wait_st(); named_bar_sync(1, 128);", {"B"}),
    ("tmem_wait_st(); if (c) fence_before(); __syncthreads();", {"B"}),
    # inline-PTX forms of the fences and operations are recognised
    ('mbar_wait(x, 0); asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); '
     'asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(t), "r"(n));', set()),
    ('mbar_wait(x, 0); asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(t), "r"(n));',
     {"A"}),
    # comments do not count
    ("mbar_wait(x, 0); // fence_after();\n mma_ss(d, a, b, i, 0);", {"A"}),
])
def test_lint_semantics_on_small_kernels(body, rules):
    src = "__global__ void __launch_bounds__(128, 1) k(int c) {\n" + body + "\n}\n"
    assert {r for _, _, r, _ in lint_source(src)} == rules
