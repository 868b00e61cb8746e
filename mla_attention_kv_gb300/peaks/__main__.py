from . import measure

print(measure())
