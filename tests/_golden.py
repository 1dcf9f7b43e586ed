"""Reader for the closed-form fixtures under tests/golden/.

Fixture values are written as small expressions (integers, + - * /, log, exp,
sqrt, -inf) and evaluated here with Python's ``decimal`` at 50 significant
digits, independently of the oracle's double arithmetic.
"""
import ast
import decimal
import os
from decimal import Decimal

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CTX = decimal.Context(prec=50)


def _eval(node):
    if isinstance(node, ast.Expression):
        return _eval(node.body)
    if isinstance(node, ast.Constant) and isinstance(node.value, (int, float)):
        return CTX.create_decimal(repr(node.value)) if isinstance(node.value, float) else Decimal(node.value)
    if isinstance(node, ast.UnaryOp) and isinstance(node.op, ast.USub):
        return -_eval(node.operand)
    if isinstance(node, ast.UnaryOp) and isinstance(node.op, ast.UAdd):
        return _eval(node.operand)
    if isinstance(node, ast.Name) and node.id == "inf":
        return Decimal("Infinity")
    if isinstance(node, ast.BinOp):
        a, b = _eval(node.left), _eval(node.right)
        op = type(node.op)
        if op is ast.Add:
            return CTX.add(a, b)
        if op is ast.Sub:
            return CTX.subtract(a, b)
        if op is ast.Mult:
            return CTX.multiply(a, b)
        if op is ast.Div:
            return CTX.divide(a, b)
    if isinstance(node, ast.Call) and isinstance(node.func, ast.Name) and len(node.args) == 1:
        v = _eval(node.args[0])
        f = node.func.id
        if f == "log":
            return CTX.ln(v)
        if f == "exp":
            return CTX.exp(v)
        if f == "sqrt":
            return CTX.sqrt(v)
    raise ValueError(f"unsupported expression node {ast.dump(node)}")


def evaluate(expr: str) -> Decimal:
    return _eval(ast.parse(expr.strip(), mode="eval"))


def read_cases(filename):
    """Yield (name, params: dict[str, Decimal], rows: dict[str, list[Decimal]])."""
    cases = []
    cur = None
    with open(os.path.join(GOLDEN, filename), encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if not line:
                continue
            if line.startswith("case "):
                parts = line.split()
                params = {}
                for p in parts[2:]:
                    k, v = p.split("=", 1)
                    params[k] = evaluate(v)
                cur = (parts[1], params, {})
                cases.append(cur)
                continue
            key, vals = line.split(":", 1)
            cur[2][key.strip()] = [evaluate(t) for t in vals.split()]
    return cases


def read_constants(filename):
    out = {}
    with open(os.path.join(GOLDEN, filename), encoding="utf-8") as f:
        for raw in f:
            line = raw.split("#", 1)[0].strip()
            if line:
                k, v = line.split()
                out[k] = v
    return out


def to_float(d: Decimal) -> float:
    return float(d)
