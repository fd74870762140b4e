"""Reader for the page-figure fixture (values printed on the source pages)."""
import os

_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "page_figures.txt")


def page_figures() -> dict:
    out = {}
    with open(_PATH, encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            kv, title, where = (part.strip() for part in line.split("|"))
            key, value = (x.strip() for x in kv.split("="))
            assert title and where, f"figure {key} has no citation"
            out[key] = float(value) if "." in value else int(value)
    return out
