"""Reader for the hand-worked fixtures under tests/golden/ (text, one
``key values...`` record per line, ``#`` comments)."""
import os

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read(name):
    records = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                key, *vals = line.split()
                records.append((key, vals))
    return records


def first(records, key):
    for k, v in records:
        if k == key:
            return v
    raise KeyError(key)


def all_of(records, key):
    return [v for k, v in records if k == key]
